// Plain SIMT GEMM (CUDA cores): Y = epilogue(X[M,K] . W[N,K]^T), f16 in, fp32 accumulate.
// Used as the in-library reference for the tensor-core GEMM's kernel tests.
// Requires K % 32 == 0; any M, N.
#include "common.cuh"

namespace s1 {

constexpr int SB = 64, SK = 32;

__device__ __forceinline__ void epilogue_store(int epi, void* out, int ldo, int M, int N, int m,
                                               int n, float v, const float* tile_row, int n_in_tile) {
  (void)tile_row; (void)n_in_tile;
  if (m >= M || n >= N) return;
  if (epi == EPI_F32) reinterpret_cast<float*>(out)[(size_t)m * ldo + n] = v;
  else if (epi == EPI_HALF) reinterpret_cast<f16*>(out)[(size_t)m * ldo + n] = f2h(v);
  else if (epi == EPI_RESADD) reinterpret_cast<float*>(out)[(size_t)m * ldo + n] += v;
}

__global__ void __launch_bounds__(256) gemm_simt_kernel(const f16* __restrict__ X,
                                                        const f16* __restrict__ W, int M, int N,
                                                        int K, int epi, void* __restrict__ out,
                                                        int ldo) {
  __shared__ float As[SK][SB + 4];
  __shared__ float Bs[SK][SB + 4];
  __shared__ float Cs[SB][SB + 1];
  const int m0 = blockIdx.y * SB, n0 = blockIdx.x * SB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // loader: 64 rows x 32 k = 2048 elements = 256 threads x 8
  const int lr = threadIdx.x >> 2, lk = (threadIdx.x & 3) * 8;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SK) {
    {
      const int m = m0 + lr;
      uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
      if (m < M) va = *reinterpret_cast<const uint4*>(X + (size_t)m * K + k0 + lk);
      const int n = n0 + lr;
      if (n < N) vb = *reinterpret_cast<const uint4*>(W + (size_t)n * K + k0 + lk);
      const f16* pa = reinterpret_cast<const f16*>(&va);
      const f16* pb = reinterpret_cast<const f16*>(&vb);
#pragma unroll
      for (int e = 0; e < 8; ++e) { As[lk + e][lr] = h2f(pa[e]); Bs[lk + e][lr] = h2f(pb[e]); }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
  __syncthreads();
  if (epi == EPI_SWIGLU) {
    // tile columns [32b, 32b+16) are gate, [32b+16, 32b+32) are up, for output columns
    // n0/2 + 16b + [0, 16).
    for (int t = threadIdx.x; t < SB * (SB / 2); t += blockDim.x) {
      const int r = t / (SB / 2), c = t % (SB / 2);
      const int b = c / 16, i = c % 16;
      const int m = m0 + r, nout = n0 / 2 + c;
      if (m < M && n0 + 32 * b + 16 + i < N) {
        const float g = Cs[r][32 * b + i], u = Cs[r][32 * b + 16 + i];
        reinterpret_cast<f16*>(out)[(size_t)m * ldo + nout] = f2h(silu_f(g) * u);
      }
    }
  } else {
    for (int t = threadIdx.x; t < SB * SB; t += blockDim.x) {
      const int r = t / SB, c = t % SB;
      epilogue_store(epi, out, ldo, M, N, m0 + r, n0 + c, Cs[r][c], nullptr, 0);
    }
  }
}

cudaError_t launch_gemm_simt(const f16* X, const f16* W, int M, int N, int K, int epi, void* out,
                             int ldo, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (K % SK) return cudaErrorInvalidValue;
  dim3 grid((N + SB - 1) / SB, (M + SB - 1) / SB);
  gemm_simt_kernel<<<grid, 256, 0, st>>>(X, W, M, N, K, epi, out, ldo);
  return cudaGetLastError();
}

}  // namespace s1
