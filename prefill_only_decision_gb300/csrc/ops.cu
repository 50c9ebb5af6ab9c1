// Kernel-level entry points (s1_ops.h): one step of the path on device pointers.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <string>
#include <vector>

#include "common.cuh"
#include "../../include/s1.h"
#include "../../include/s1_ops.h"

using namespace s1;

namespace s1 {
int set_error(int code, const char* msg);   // s1_api.cu: the thread-local message of s1_last_error
}

namespace {
int op_fail(int code, const char* msg) { return s1::set_error(code, msg); }
#define OCK(call)                                                                            \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess) {                                                                 \
      char b_[256];                                                                          \
      snprintf(b_, sizeof(b_), "%s: %s", #call, cudaGetErrorString(e_));                     \
      return op_fail(S1_ERR_CUDA, b_);                                                       \
    }                                                                                        \
  } while (0)

struct Tmp {
  std::vector<void*> ps;
  ~Tmp() { for (void* p : ps) cudaFree(p); }
  void* get(size_t b) {
    void* p = nullptr;
    if (cudaMalloc(&p, b ? b : 16) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    ps.push_back(p);
    return p;
  }
};
}  // namespace

extern "C" {

int s1_op_gemm(const void* X, const void* W, int32_t M, int32_t N, int32_t K, int32_t epi, void* out,
               int32_t ldo, int32_t impl, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (M < 0 || N <= 0 || K <= 0 || K % 64 || N % 32 || epi < 0 || epi > 3)
    return op_fail(S1_ERR_INVALID_ARG, "gemm: bad sizes or epilogue");
  Tmp t;
  if (impl < 0 || impl > 3) return op_fail(S1_ERR_INVALID_ARG, "gemm: impl must be 0..3");
  if (impl != 1) {
    if (!gemm_tc_supported(M, N, K, epi)) return op_fail(S1_ERR_UNSUPPORTED, "gemm: shape not supported by the tensor-core kernel");
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t wsf = gemm_tc_workspace_floats(M, N, K, epi, sms);
    float* ws = (float*)t.get(wsf * 4 + 16);
    int* err = (int*)t.get(256);
    if (!ws || !err) return op_fail(S1_ERR_OOM, "gemm: temporaries");
    OCK(cudaMemsetAsync(err, 0, 256, st));
    LaunchCtx lc{st, err, sms, nullptr};
    lc.variant = impl == 2 ? GEMM_PAIR : (impl == 3 ? GEMM_SINGLE : GEMM_ANY);
    OCK(launch_gemm_tc((const f16*)X, (const f16*)W, M, N, K, epi, out, ldo, ws, wsf, lc));
    int h = 0;
    OCK(cudaMemcpyAsync(&h, err, 4, cudaMemcpyDeviceToHost, st));
    OCK(cudaStreamSynchronize(st));
    if (h) return op_fail(S1_ERR_DEVICE_TIMEOUT, "gemm: a bounded device wait gave up");
    return S1_OK;
  }
  OCK(launch_gemm_simt((const f16*)X, (const f16*)W, M, N, K, epi, out, ldo, st));
  OCK(cudaStreamSynchronize(st));
  return S1_OK;
}

int s1_op_gdn(float* proj, int32_t R, int32_t H, int32_t dk, int32_t dv, float l2_eps, int32_t n_seq,
              const int32_t* row0, const int32_t* len, const float* S0, float* S_out, void* out,
              void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (R < 0 || H <= 0 || n_seq <= 0 || !row0 || !len) return op_fail(S1_ERR_INVALID_ARG, "gdn: bad arguments");
  std::vector<SeqDesc> seqs(n_seq);
  std::vector<CtxDesc> ctxs(2 * n_seq);
  std::vector<ChunkDesc> chunks;
  const size_t per = (size_t)H * dv * dk;
  for (int s = 0; s < n_seq; ++s) {
    if (row0[s] < 0 || len[s] < 0 || row0[s] + len[s] > R) return op_fail(S1_ERR_INVALID_ARG, "gdn: sequence outside rows");
    seqs[s] = SeqDesc{row0[s], len[s], 0, S0 ? s : -1, S_out ? n_seq + s : -1, (int)chunks.size()};
    for (int c = 0; c < len[s]; c += GDN_CHUNK)
      chunks.push_back(ChunkDesc{row0[s] + c, len[s] - c < GDN_CHUNK ? len[s] - c : GDN_CHUNK, s});
    ctxs[s] = CtxDesc{const_cast<float*>(S0 ? S0 + s * per : nullptr), nullptr, 0, 0};
    ctxs[n_seq + s] = CtxDesc{S_out ? S_out + s * per : nullptr, nullptr, 0, 0};
  }
  const int nch = (int)chunks.size();
  Tmp t;
  SeqDesc* dseq = (SeqDesc*)t.get(seqs.size() * sizeof(SeqDesc));
  CtxDesc* dctx = (CtxDesc*)t.get(ctxs.size() * sizeof(CtxDesc));
  ChunkDesc* dch = (ChunkDesc*)t.get((nch + 1) * sizeof(ChunkDesc));
  float* loga = (float*)t.get((size_t)R * H * 4 + 16);
  float* beta = (float*)t.get((size_t)R * H * 4 + 16);
  if (!dseq || !dctx || !dch || !loga || !beta) return op_fail(S1_ERR_OOM, "gdn: temporaries");
  OCK(cudaMemcpyAsync(dseq, seqs.data(), seqs.size() * sizeof(SeqDesc), cudaMemcpyHostToDevice, st));
  OCK(cudaMemcpyAsync(dctx, ctxs.data(), ctxs.size() * sizeof(CtxDesc), cudaMemcpyHostToDevice, st));
  if (nch) OCK(cudaMemcpyAsync(dch, chunks.data(), nch * sizeof(ChunkDesc), cudaMemcpyHostToDevice, st));
  const int ld = 2 * H * dk + H * dv + 2 * H;
  if (gdn_chunked_supported(H, dk, dv, ld)) {   // normalisation and gates inside the chunked kernels
    void* rows = t.get((size_t)R * gdn_row_bytes(H, dk) + 16);
    void* per_chunk = t.get((size_t)nch * gdn_chunk_bytes(H, dk) + 16);
    int* err = (int*)t.get(256);
    if (!rows || !per_chunk || !err) return op_fail(S1_ERR_OOM, "gdn: temporaries");
    OCK(cudaMemsetAsync(err, 0, 256, st));
    int dev = 0, sms = 0;
    OCK(cudaGetDevice(&dev));
    OCK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const GdnBufs gb = gdn_bufs(rows, (size_t)R, per_chunk, (size_t)nch, H, dk);
    OCK(launch_gdn_chunked(proj, ld, loga, l2_eps, (f16*)out, dseq, n_seq, dch, nch, dctx, 0, H, dk, dv, gb, 0, n_seq,
                           n_seq, err, sms, st, nullptr));
    int herr = 0;
    OCK(cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st));
    OCK(cudaStreamSynchronize(st));
    if (herr) return op_fail(S1_ERR_DEVICE_TIMEOUT, "gdn: a bounded device wait gave up");
  } else {
    OCK(launch_gdn_prep(proj, ld, loga, beta, R, H, dk, dv, l2_eps, st));
    OCK(launch_gdn_scan(proj, ld, loga, beta, (f16*)out, dseq, n_seq, dctx, 0, H, dk, dv, st));
  }
  OCK(cudaStreamSynchronize(st));
  return S1_OK;
}

int s1_op_attention(const void* q, const void* k_new, const void* v_new, const void* kv_cache, int32_t P,
                    int32_t n_seq, const int32_t* row0, const int32_t* len, int32_t Hq, int32_t Hkv,
                    int32_t hd, void* out, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (n_seq <= 0 || !row0 || !len || P < 0 || (P > 0 && !kv_cache) || Hq % Hkv)
    return op_fail(S1_ERR_INVALID_ARG, "attention: bad arguments");
  std::vector<SeqDesc> seqs(n_seq);
  int max_len = 0;
  for (int s = 0; s < n_seq; ++s) {
    seqs[s] = SeqDesc{row0[s], len[s], P, P > 0 ? 0 : -1, -1, 0};
    max_len = len[s] > max_len ? len[s] : max_len;
  }
  CtxDesc c{nullptr, (f16*)kv_cache, P, P};
  Tmp t;
  SeqDesc* dseq = (SeqDesc*)t.get(seqs.size() * sizeof(SeqDesc));
  CtxDesc* dctx = (CtxDesc*)t.get(sizeof(CtxDesc));
  if (!dseq || !dctx) return op_fail(S1_ERR_OOM, "attention: temporaries");
  OCK(cudaMemcpyAsync(dseq, seqs.data(), seqs.size() * sizeof(SeqDesc), cudaMemcpyHostToDevice, st));
  OCK(cudaMemcpyAsync(dctx, &c, sizeof(CtxDesc), cudaMemcpyHostToDevice, st));
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int R = 0;
  for (int i = 0; i < n_seq; ++i) R = std::max(R, row0[i] + len[i]);
  const char* ga = getenv("S1_ATTN");   // "sync": the mma.sync kernel (debugging)
  if (!(ga && strcmp(ga, "sync") == 0) && attention_tc_supported(hd)) {
    // the tensor-core kernel: the cache as one context of one layer ([2, P, Hkv, hd])
    long work_ctas = 0;
    for (int i = 0; i < n_seq; ++i) work_ctas += (long)((len[i] + 127) / 128) * Hq;
    std::vector<uint8_t> map(attention_ctx_map_bytes(), 0);
    if (P > 0 && !attention_ctx_map(map.data(), (const f16*)kv_cache, 1, P, P, Hkv, hd))
      return op_fail(S1_ERR_CUDA, "attention: tensor map encoding failed");
    void* dmap = t.get(map.size() + 128);
    int* err = (int*)t.get(256);
    if (!dmap || !err) return op_fail(S1_ERR_OOM, "attention: temporaries");
    dmap = (void*)(((uintptr_t)dmap + 127) & ~(uintptr_t)127);
    OCK(cudaMemcpyAsync(dmap, map.data(), map.size(), cudaMemcpyHostToDevice, st));
    OCK(cudaMemsetAsync(err, 0, 256, st));
    OCK(launch_attention_tc((const f16*)q, (const f16*)k_new, (const f16*)v_new, (f16*)out, R, dseq, n_seq, dctx,
                            dmap, 0, Hq, Hkv, hd, max_len, P + max_len, work_ctas, sms, err, st));
    int herr = 0;
    OCK(cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st));
    OCK(cudaStreamSynchronize(st));
    if (herr) return op_fail(S1_ERR_DEVICE_TIMEOUT, "attention: a bounded device wait gave up");
    return S1_OK;
  }
  long work_ctas = 0;
  for (int i = 0; i < n_seq; ++i) work_ctas += (long)((len[i] + 63) / 64) * Hq;
  OCK(launch_attention((const f16*)q, (const f16*)k_new, (const f16*)v_new, (f16*)out, dseq, n_seq,
                       dctx, 0, Hq, Hkv, hd, max_len, P + max_len, work_ctas, sms, st));
  OCK(cudaStreamSynchronize(st));
  return S1_OK;
}

int s1_op_rmsnorm(const float* x, const float* w, int32_t R, int32_t d, float eps, void* out, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (R < 0 || d <= 0 || d % 4) return op_fail(S1_ERR_INVALID_ARG, "rmsnorm: bad sizes");
  OCK(launch_rmsnorm(x, w, (f16*)out, R, d, eps, st));
  OCK(cudaStreamSynchronize(st));
  return S1_OK;
}

}  // extern "C"
