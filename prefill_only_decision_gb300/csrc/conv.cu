// Short causal convolution of the gated delta-rule layers (the snapshot's "convolution history",
// System1-Omni RFC #114, section 5): each q | k | v channel of the in-projection is convolved
// causally over a sequence's rows with its own W taps, then passed through SiLU, before the
// gated delta rule normalises q and k.
//   y_i[c] = SiLU( sum_{j < W} w[c][j] * x_{i - (W-1) + j}[c] )
// Rows before the sequence's first come from the W - 1 rows of history of the snapshot it
// continues (zeros at a fresh start); a sequence that writes a snapshot leaves its own last W - 1
// input rows there. One thread per (row, 4 channels); the a | b gate columns are copied.
#include "common.cuh"

namespace s1 {

__global__ void __launch_bounds__(256) short_conv_kernel(const float* __restrict__ x, float* __restrict__ out,
                                                         int ld, int channels, const float* __restrict__ w, int W,
                                                         const SeqDesc* __restrict__ seqs,
                                                         const CtxDesc* __restrict__ ctxs, int layer_g) {
  allow_dependents();
  wait_prerequisites();
  const SeqDesc sd = seqs[blockIdx.y];
  const int q4 = ld / 4;
  const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const int i = (int)(t / q4), c = (int)(t % q4) * 4;
  const bool conv_row = i < sd.len;                              // an output row of the sequence
  const bool hist_row = sd.ctx_out >= 0 && W > 1 && i < W - 1;   // a history row it writes
  if (!conv_row && !hist_row) return;
  const size_t row = (size_t)(sd.row0 + i) * ld;
  if (c >= channels) {   // gate inputs a | b: unchanged
    if (conv_row) *reinterpret_cast<float4*>(out + row + c) = *reinterpret_cast<const float4*>(x + row + c);
    return;
  }
  const size_t hstride = (size_t)(W - 1) * channels;   // history floats per layer
  const float* hin = (sd.ctx_in >= 0 && ctxs[sd.ctx_in].conv) ? ctxs[sd.ctx_in].conv + layer_g * hstride : nullptr;
  // input row m of the sequence (m < 0: the history it continues)
  auto X = [&](int m) -> float4 {
    if (m >= 0) return *reinterpret_cast<const float4*>(x + (size_t)(sd.row0 + m) * ld + c);
    if (!hin) return make_float4(0.f, 0.f, 0.f, 0.f);
    return *reinterpret_cast<const float4*>(hin + (size_t)(W - 1 + m) * channels + c);
  };
  if (conv_row) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < W; ++j) {
      const float4 v = X(i - (W - 1) + j);
      acc.x = fmaf(w[(size_t)c * W + j], v.x, acc.x);
      acc.y = fmaf(w[(size_t)(c + 1) * W + j], v.y, acc.y);
      acc.z = fmaf(w[(size_t)(c + 2) * W + j], v.z, acc.z);
      acc.w = fmaf(w[(size_t)(c + 3) * W + j], v.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + row + c) =
        make_float4(silu_f(acc.x), silu_f(acc.y), silu_f(acc.z), silu_f(acc.w));
  }
  // the snapshot's new history: the last W - 1 input rows, reaching into the old history when
  // the sequence is shorter (history row k = input row len - (W-1) + k, written by thread row k)
  if (hist_row) {
    float* hout = ctxs[sd.ctx_out].conv;
    if (hout) *reinterpret_cast<float4*>(hout + layer_g * hstride + (size_t)i * channels + c) = X(sd.len - (W - 1) + i);
  }
}

cudaError_t launch_short_conv(const float* x, float* out, int ld, int channels, const float* w, int W,
                              const SeqDesc* d_seq, int seq0, int n_seq, int max_len, const CtxDesc* d_ctx,
                              int layer_g, cudaStream_t st) {
  if (n_seq <= 0 || max_len <= 0) return cudaSuccess;
  if (ld % 4 || channels % 4 || channels > ld || W < 1 || n_seq > 65535) return cudaErrorInvalidValue;
  const long threads = (long)(max_len > W - 1 ? max_len : W - 1) * (ld / 4);
  const dim3 grid((unsigned)((threads + 255) / 256), n_seq);
  CK_RET(launch_pdl(short_conv_kernel, grid, dim3(256), 0, st, x, out, ld, channels, w, W, d_seq + seq0, d_ctx,
                    layer_g));
  return cudaGetLastError();
}

}  // namespace s1
