// Causal GQA attention over packed sequences, with suffix-over-prefix continuation.
//
// A query at row i of sequence s (position pos0 + i) attends to every cached key of the
// snapshot it continues (positions 0 .. P-1) and to its own sequence's keys 0 .. i; never
// to another sequence ("execute isolated question/option suffixes", System1-Omni RFC #114,
// section 4, "Branching" row). q head h reads kv head floor(h * Hkv / Hq).
// softmax(q.k / sqrt(hd)) v with an online (running max / sum) softmax in fp32.
#include "common.cuh"

namespace s1 {

// One warp per (row, q head); a lane holds hd/32 consecutive dims.
template <int HD>
__global__ void __launch_bounds__(128) attn_rowwarp_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ knew, const bf16* __restrict__ vnew,
    bf16* __restrict__ out, const SeqDesc* __restrict__ seqs, const CtxDesc* __restrict__ ctxs,
    int layer_f, int Hq, int Hkv, float scale_log2) {
  constexpr int E = HD / 32;
  const int sq = blockIdx.y;
  const SeqDesc sd = seqs[sq];
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + (threadIdx.x >> 5);   // (row, head) within the sequence
  if (item >= sd.len * Hq) return;
  const int i = item / Hq, h = item % Hq;
  const int g = (h * Hkv) / Hq;
  const int row = sd.row0 + i;
  float qv[E];
  const bf16* qp = q + ((size_t)row * Hq + h) * HD + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) qv[e] = bf2f(qp[e]) * scale_log2;
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  auto visit = [&](const bf16* kp, const bf16* vp) {
    float sdot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) sdot = fmaf(qv[e], bf2f(kp[e]), sdot);
    sdot = warp_sum(sdot);
    const float mn = fmaxf(m, sdot);
    const float c = exp2f(m - mn), p = exp2f(sdot - mn);
    l = l * c + p;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(acc[e], c, p * bf2f(vp[e]));
    m = mn;
  };
  if (sd.ctx_in >= 0) {
    const CtxDesc c = ctxs[sd.ctx_in];
    const size_t plane = (size_t)c.cap * Hkv * HD;
    const bf16* Kc = c.KV + (size_t)layer_f * 2 * plane + (size_t)g * HD + lane * E;
    const bf16* Vc = Kc + plane;
    for (int j = 0; j < c.P; ++j) visit(Kc + (size_t)j * Hkv * HD, Vc + (size_t)j * Hkv * HD);
  }
  const bf16* Kn = knew + ((size_t)sd.row0 * Hkv + g) * HD + lane * E;
  const bf16* Vn = vnew + ((size_t)sd.row0 * Hkv + g) * HD + lane * E;
  for (int j = 0; j <= i; ++j) visit(Kn + (size_t)j * Hkv * HD, Vn + (size_t)j * Hkv * HD);
  const float inv = 1.f / l;
  bf16* op = out + ((size_t)row * Hq + h) * HD + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) op[e] = f2bf(acc[e] * inv);
}

cudaError_t launch_attention(const bf16* q, const bf16* knew, const bf16* vnew, bf16* out,
                             const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx, int layer_f,
                             int Hq, int Hkv, int hd, int max_len, cudaStream_t st) {
  if (n_seq <= 0 || max_len <= 0) return cudaSuccess;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  dim3 grid((max_len * Hq + 3) / 4, n_seq);
  if (hd == 128)
    attn_rowwarp_kernel<128><<<grid, 128, 0, st>>>(q, knew, vnew, out, d_seq, d_ctx, layer_f, Hq, Hkv, scale_log2);
  else if (hd == 64)
    attn_rowwarp_kernel<64><<<grid, 128, 0, st>>>(q, knew, vnew, out, d_seq, d_ctx, layer_f, Hq, Hkv, scale_log2);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

}  // namespace s1
