// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace s1 {

// bf16: the model's stored tensors as the caller gives them (embedding table, given embedding
// rows, bf16 weight arrays). f16: every tensor-core operand of the forward pass (merged weights,
// normed rows, mixer and MLP outputs, attention q/k/v and the K/V snapshot): the same tensor-core
// rate as bf16 with three more mantissa bits (bf16 weights convert to f16 exactly down to 2^-14,
// and below it to within 2^-25).
typedef __nv_bfloat16 bf16;
typedef __half f16;

// GEMM epilogues: Y = X[M,K] . W[N,K]^T accumulated in fp32, then
enum Epilogue {
  EPI_F32 = 0,      // out fp32 [M, ldo]: out = acc
  EPI_HALF = 1,     // out f16 [M, ldo]: out = f16(acc)
  EPI_RESADD = 2,   // out fp32 [M, ldo]: out += acc   (residual stream)
  EPI_SWIGLU = 3,   // W rows interleaved in blocks of 16 gate / 16 up rows;
                    // out f16 [M, ldo] with N/2 columns: silu(gate) * up
  EPI_LSE = 4,      // out float2 [ceil(N / BN), ldo]: per row m and N tile t, (max, sum of
                    // exp(acc - max)) over the tile's columns (launch_gemm_lse only)
};

// Packed description of the sequences of one forward call.
struct SeqDesc {
  int row0;     // first packed row
  int len;      // rows
  int pos0;     // position of the first row
  int ctx_in;   // context continued (-1: start from zero state / no cached keys)
  int ctx_out;  // context whose snapshot this sequence writes (-1: none)
  int chunk0;   // index of its first 64-row chunk in the chunk table
  int fol0, fol1;   // gated delta rule: single-chunk sequences [fol0, fol1) that continue from this
                    // one's final state and keep none of their own (their U and chunk-start state
                    // come from this sequence's state pass; empty if fol1 <= fol0)
};

// 64-row chunks of the sequences (chunk boundaries restart at every sequence start).
struct ChunkDesc {
  int row0;
  int len;      // 1 .. 64
  int seq;
};
constexpr int GDN_CHUNK = 64;

// A prefix snapshot as seen by kernels: all layers' tensors of one state.
struct CtxDesc {
  float* S;     // [n_gdn_layers, H, Dv, Dk] fp32
  f16* KV;      // [n_fa_layers, 2, cap, Hkv, hd] f16
  int P;        // cached rows
  int cap;      // capacity rows
  float* conv = nullptr;   // short-convolution history [n_gdn_layers, width - 1, channels] fp32
};

// GEMM kernel families a launch may choose from.
enum { GEMM_ANY = 0, GEMM_SINGLE = 1, GEMM_PAIR = 2 };

struct LaunchCtx {
  cudaStream_t stream;
  int* d_err;        // device error word (bounded waits record here)
  int num_sms;
  long* launches;    // incremented per kernel launched (may be NULL)
  bool tune = false;          // GEMM: measure the tile choice on first use of a shape
  void* tune_out = nullptr;   // GEMM tuning: scratch output for residual-add shapes (fp32)
  size_t tune_floats = 0;
  void* tune_flush = nullptr; // GEMM tuning: buffer larger than L2, rewritten before each timed run
  size_t tune_flush_bytes = 0;
  int variant = GEMM_ANY;     // GEMM: kernel families allowed (GEMM_ANY, GEMM_SINGLE, GEMM_PAIR)
  // GEMM, residual add with a K split over at most 512 rows: the RMSNorm of the updated rows,
  // out = f16(x / sqrt(mean(x^2) + norm_eps) * norm_w), fused into the split-K reduction
  // (same arithmetic and order as launch_rmsnorm over that many rows, so the same bits).
  const float* norm_w = nullptr;   // [N] fp32; NULL: no fused norm
  f16* norm_out = nullptr;         // [M, N] f16
  float norm_eps = 0.f;
  bool* norm_done = nullptr;       // set to true when the norm was fused (the caller skips its own)
};

// Threads of a block that normalises one row of width d (one float4 per thread and pass): the
// block-per-row RMSNorm and the split-K reduction that fuses it use the same count, so that
// their sums run in the same order.
inline int norm_row_threads(int d) {
  const int t = ((d / 4 + 31) / 32) * 32;
  return t < 32 ? 32 : (t > 1024 ? 1024 : t);
}

// Tiled TMA descriptor over a global tensor (dims and box innermost first, strides in bytes for
// dims 1..rank-1), encoded through the driver entry point and cached by its arguments.
// Returns false if the driver entry point is missing or rejects the arguments.
bool tensor_map(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* ptr, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle);

// ---- kernels (launchers) ----
cudaError_t launch_embed(const f16* E, const int* row_src, const bf16* embeds, float* x, int R, int d,
                         cudaStream_t st);
cudaError_t launch_rmsnorm(const float* x, const float* w, f16* out, int R, int d, float eps,
                           cudaStream_t st);
cudaError_t launch_gemm_simt(const f16* X, const f16* W, int M, int N, int K, int epi, void* out,
                             int ldo, cudaStream_t st);
bool gemm_tc_supported(int M, int N, int K, int epi);
cudaError_t launch_gemm_tc(const f16* X, const f16* W, int M, int N, int K, int epi, void* out,
                           int ldo, float* splitk_ws, size_t ws_floats, const LaunchCtx& lc);
// Row-wise log-sum-exp partials of X . W^T on the tensor cores (no K split, 256-wide N tiles):
// part[t * ldp + m] = (max, sum exp(acc - max)) over the columns of N tile t, for m < M <= ldp.
constexpr int GEMM_LSE_BN = 256;
cudaError_t launch_gemm_lse(const f16* X, const f16* W, int M, int N, int K, float2* part, int ldp,
                            const LaunchCtx& lc);
size_t gemm_tc_workspace_floats(int M, int N, int K, int epi, int num_sms);
size_t gemm_tc_plan_ws_floats(int M, int N, int K, int epi, int num_sms, size_t ws_cap);
cudaError_t launch_gdn_prep(float* proj, int ld, float* alpha, float* beta, int R, int H, int Dk,
                            int Dv, float eps, cudaStream_t st);
cudaError_t launch_gdn_scan(const float* proj, int ld, const float* alpha, const float* beta,
                            f16* out, const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx,
                            int layer_g, int H, int Dk, int Dv, cudaStream_t st);
bool gdn_chunked_supported(int H, int Dk, int Dv, int ld);
// Scratch of the chunked gated delta rule (D = dk = dv): per packed row and head, the normalised
// k, W, Ut and the decayed keys K' (f16 [R, H, D] each); per chunk and head, N^T = (W^T K')^T
// (f16 [D, D]), the chunk's start state (f16 [D, D]) and its total decay gamma_n (fp32).
struct GdnBufs {
  f16* Kn;
  f16* W;
  f16* Ut;
  f16* Kp;
  f16* NT;
  f16* Srec;
  float* gam;
  size_t rows;                          // R of the per-row arrays
  size_t n_chunks_cap;
};
size_t gdn_row_bytes(int H, int D);     // bytes per packed row
size_t gdn_chunk_bytes(int H, int D);   // bytes per chunk
GdnBufs gdn_bufs(void* rows, size_t R, void* per_chunk, size_t n_chunks, int H, int D);
cudaError_t launch_gdn_chunked(const float* proj, int ld, float* gbuf, float l2_eps, f16* out, const SeqDesc* d_seq,
                               int n_seq, const ChunkDesc* d_chunks, int n_chunks, const CtxDesc* d_ctx, int layer_g,
                               int H, int Dk, int Dv, const GdnBufs& bufs, int n_first, int fold_from, int out_fold,
                               int* d_err, int num_sms, cudaStream_t st, long* launches);
cudaError_t launch_rope_split(const float* proj, int ld, const float2* rope_tab, const int* row_seq,
                              const SeqDesc* d_seq, const CtxDesc* d_ctx, int layer_f, f16* q,
                              f16* knew, f16* vnew, int R, int Hq, int Hkv, int hd,
                              cudaStream_t st);
cudaError_t launch_attention(const f16* q, const f16* knew, const f16* vnew, f16* out,
                             const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx, int layer_f,
                             int Hq, int Hkv, int hd, int max_len, int max_keys, long work_ctas, int num_sms,
                             cudaStream_t st);
// Attention on tcgen05 (head dims 64 and 128). d_ctx_maps: device array of tensor maps, one per
// context of the call (attention_ctx_map over its snapshot's K/V; 64-byte aligned entries of
// attention_ctx_map_bytes() bytes). R: rows of q / knew / vnew.
bool attention_tc_supported(int hd);
size_t attention_ctx_map_bytes();
bool attention_ctx_map(void* map_out, const f16* kv, int n_fa_layers, int P, int cap, int Hkv, int hd);
cudaError_t launch_attention_tc(const f16* q, const f16* knew, const f16* vnew, f16* out, int R,
                                const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx, const void* d_ctx_maps,
                                int layer_f, int Hq, int Hkv, int hd, int max_len, int max_keys, long work_ctas,
                                int num_sms, int* d_err, cudaStream_t st);
cudaError_t launch_readout(const float* x, const float* final_norm, const f16* E, int d, float eps,
                           const int* q_row, const int* q_type, const int* opt_off,
                           const int* opt_ids, int n_q, float* probs, float* stats, float* hidden,
                           int max_opts, float* hn_out, float* z_out, cudaStream_t st);
size_t vocab_lm_scratch_floats(int n_q, int n_opts, int d, int V, int num_sms);
cudaError_t launch_vocab_lm(const f16* E, int V, int d, const float* hn, const float* z, const int* opt_off, int n_q,
                            float* lm, float* scratch, const LaunchCtx& lc, bool tensor_cores);
cudaError_t launch_merge_lora(const void* W, int w_is_bf16, const void* A, const void* B,
                              int ab_is_bf16, int rank, float scale, int out_f, int in_f,
                              f16* dst, int dst_row0, int interleave_swiglu, int swiglu_half,
                              int swiglu_F, float* tmpA, float* tmpB, cudaStream_t st);
cudaError_t launch_to_f32(const void* src, int is_bf16, float* dst, size_t n, cudaStream_t st);
// Short causal convolution of the gated delta-rule layers: out[:, c] = SiLU(sum_j w[c][j] *
// x[row - (W-1) + j, c]) over the first `channels` columns of each row (q | k | v), the rows
// before a sequence's start taken from its snapshot's history (ctx_in, else zeros); the a | b
// columns [channels, ld) are copied. Sequences that write a snapshot (ctx_out) store their last
// W - 1 input rows as its history. w: fp32 [channels, W]. One launch covers sequences
// [seq0, seq0 + n_seq); rows of other sequences are left alone.
cudaError_t launch_short_conv(const float* x, float* out, int ld, int channels, const float* w, int W,
                              const SeqDesc* d_seq, int seq0, int n_seq, int max_len, const CtxDesc* d_ctx,
                              int layer_g, cudaStream_t st);
cudaError_t launch_rope_table(float2* tab, int max_pos, int hd, double theta, cudaStream_t st);

}  // namespace s1
