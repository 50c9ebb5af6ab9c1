// Full-vocabulary log-probabilities of the option tokens at each question's readout row:
// log p(o) = z_o - log sum_v exp(z_v), z = E h_hat with E the tied embedding [V, d]
// (System1-Omni RFC #114, section 4 "Readout" row and the paragraph after the table: token
// log-probabilities normalised over the full vocabulary, computed in bounded vocabulary chunks).
// Tensor-core pass (the default): z = E h_hat for all questions at once is a [n_q, V] x d
// contraction, run on the tcgen05 GEMM with h_hat rounded to f16; its epilogue reduces each row's
// 256 logits of an N tile to a (max, sum of exp) pair, so no logit is ever stored, and E streams
// from HBM once per 128 questions. CUDA-core pass (vocabularies that are not a multiple of 32, or
// S1_VOCAB=simt): every CTA owns a block of vocabulary rows and keeps a running (max, sum of exp)
// per question in fp32 over groups of up to QG questions. Either way a second kernel combines the
// partials in a fixed order, and lm[o] = z_o - lse with z_o the readout's fp32 option logit.
#include <algorithm>
#include "common.cuh"

namespace s1 {

template <int QG>
__global__ void __launch_bounds__(256) vocab_lse_kernel(const f16* __restrict__ E, int V, int d,
                                                        const float* __restrict__ hn, int n_q, int rows_per_block,
                                                        float2* __restrict__ part) {
  extern __shared__ float hs[];   // [QG][d] normalised readout rows of the current group
  __shared__ float2 wred[8][QG];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = blockIdx.x * rows_per_block;
  const int r1 = min(V, r0 + rows_per_block);
  for (int q0 = 0; q0 < n_q; q0 += QG) {
    const int qn = min(QG, n_q - q0);
    __syncthreads();
    for (int i = threadIdx.x; i < QG * d; i += blockDim.x) {
      const int q = i / d;
      hs[i] = q < qn ? hn[(size_t)(q0 + q) * d + (i % d)] : 0.f;
    }
    __syncthreads();
    float m[QG], s[QG];
#pragma unroll
    for (int q = 0; q < QG; ++q) { m[q] = -INFINITY; s[q] = 0.f; }
    for (int r = r0 + warp; r < r1; r += 8) {
      const uint4* er = reinterpret_cast<const uint4*>(E + (size_t)r * d);
      float acc[QG];
#pragma unroll
      for (int q = 0; q < QG; ++q) acc[q] = 0.f;
      for (int c = lane; c < d / 8; c += 32) {
        const uint4 e = er[c];
        const f16* eb = reinterpret_cast<const f16*>(&e);
        float ef[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ef[i] = h2f(eb[i]);
#pragma unroll
        for (int q = 0; q < QG; ++q) {
          const float4 h0 = *reinterpret_cast<const float4*>(&hs[q * d + 8 * c]);
          const float4 h1 = *reinterpret_cast<const float4*>(&hs[q * d + 8 * c + 4]);
          acc[q] += ef[0] * h0.x + ef[1] * h0.y + ef[2] * h0.z + ef[3] * h0.w + ef[4] * h1.x + ef[5] * h1.y +
                    ef[6] * h1.z + ef[7] * h1.w;
        }
      }
#pragma unroll
      for (int q = 0; q < QG; ++q) {
        const float z = warp_sum(acc[q]);
        const float mn = fmaxf(m[q], z);
        s[q] = s[q] * __expf(m[q] - mn) + __expf(z - mn);
        m[q] = mn;
      }
    }
    if (lane == 0)
#pragma unroll
      for (int q = 0; q < QG; ++q) wred[warp][q] = make_float2(m[q], s[q]);
    __syncthreads();
    if (threadIdx.x < qn) {
      const int q = threadIdx.x;
      float mm = -INFINITY;
      for (int w = 0; w < 8; ++w) mm = fmaxf(mm, wred[w][q].x);
      float ss = 0.f;
      for (int w = 0; w < 8; ++w)
        if (wred[w][q].x > -INFINITY) ss += wred[w][q].y * __expf(wred[w][q].x - mm);
      part[(size_t)blockIdx.x * n_q + q0 + q] = make_float2(mm, ss);
    }
  }
}

// lse per question from the per-block partials (fixed order); lm[o] = z[o] - lse for its options.
__global__ void vocab_finish_kernel(const float2* __restrict__ part, int n_blocks, int n_q,
                                    const int* __restrict__ opt_off, const float* __restrict__ z,
                                    float* __restrict__ lm, float* __restrict__ lse_out) {
  const int q = blockIdx.x;
  __shared__ float red[32];
  __shared__ float s_lse;
  float mm = -INFINITY;
  for (int b = threadIdx.x; b < n_blocks; b += blockDim.x) mm = fmaxf(mm, part[(size_t)b * n_q + q].x);
  // block max
  mm = warp_max(mm);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mm;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float M = red[0];
  __syncthreads();
  float ss = 0.f;
  for (int b = threadIdx.x; b < n_blocks; b += blockDim.x) {
    const float2 p = part[(size_t)b * n_q + q];
    if (p.x > -INFINITY) ss += p.y * __expf(p.x - M);
  }
  ss = block_sum(ss, red);
  if (threadIdx.x == 0) {
    s_lse = M + logf(ss);
    if (lse_out) lse_out[q] = s_lse;
  }
  __syncthreads();
  for (int o = opt_off[q] + threadIdx.x; o < opt_off[q + 1]; o += blockDim.x) lm[o] = z[o] - s_lse;
}

__global__ void to_half_kernel(const float* __restrict__ x, f16* __restrict__ y, size_t n) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = f2h(x[i]);
}

static int cuda_core_blocks(int num_sms) { return 4 * (num_sms > 0 ? num_sms : 152); }

size_t vocab_lm_scratch_floats(int n_q, int n_opts, int d, int V, int num_sms) {
  const size_t tiles = (size_t)(V + GEMM_LSE_BN - 1) / GEMM_LSE_BN;
  const size_t parts = std::max(tiles, (size_t)cuda_core_blocks(num_sms));
  // h_hat fp32 | h_hat f16 (128-byte aligned) | partial pairs
  return (size_t)n_opts + (size_t)n_q * d + ((size_t)n_q * d + 1) / 2 + 64 + parts * n_q * 2 + 64;
}

cudaError_t launch_vocab_lm(const f16* E, int V, int d, const float* hn, const float* z, const int* opt_off, int n_q,
                            float* lm, float* scratch, const LaunchCtx& lc, bool tensor_cores) {
  if (n_q <= 0) return cudaSuccess;
  cudaStream_t st = lc.stream;
  if (tensor_cores && gemm_tc_supported(n_q, V, d, EPI_F32)) {
    f16* h16 = reinterpret_cast<f16*>(((uintptr_t)scratch + 127) & ~(uintptr_t)127);
    const size_t nh = (size_t)n_q * d;
    float2* part = reinterpret_cast<float2*>(((uintptr_t)(h16 + nh) + 127) & ~(uintptr_t)127);
    to_half_kernel<<<(unsigned)((nh + 255) / 256), 256, 0, st>>>(hn, h16, nh);
    CK_RET(cudaGetLastError());
    CK_RET(launch_gemm_lse(h16, E, n_q, V, d, part, n_q, lc));
    const int tiles = (V + GEMM_LSE_BN - 1) / GEMM_LSE_BN;
    vocab_finish_kernel<<<n_q, 256, 0, st>>>(part, tiles, n_q, opt_off, z, lm, nullptr);
    if (lc.launches) *lc.launches += 2;   // (the GEMM counts its own launch)
    return cudaGetLastError();
  }
  const int blocks = cuda_core_blocks(lc.num_sms);
  const int rows_per_block = (V + blocks - 1) / blocks;
  float2* part = reinterpret_cast<float2*>(((uintptr_t)scratch + 127) & ~(uintptr_t)127);
  const int qg = (d * 4 * 8 <= 96 * 1024) ? 8 : 4;
  const size_t smem = (size_t)qg * d * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(vocab_lse_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(vocab_lse_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  if (qg == 8) vocab_lse_kernel<8><<<blocks, 256, smem, st>>>(E, V, d, hn, n_q, rows_per_block, part);
  else vocab_lse_kernel<4><<<blocks, 256, smem, st>>>(E, V, d, hn, n_q, rows_per_block, part);
  vocab_finish_kernel<<<n_q, 256, 0, st>>>(part, blocks, n_q, opt_off, z, lm, nullptr);
  if (lc.launches) *lc.launches += 2;
  return cudaGetLastError();
}

}  // namespace s1
