// Chunked gated delta rule (WY form) for prefill-length sequences.
//
// For a chunk of n <= 64 rows with state S0 at its start ([Dv, Dk] per head), with
// g = cumsum(log alpha) inside the chunk, gamma = exp(g), Gamma_ts = exp(g_t - g_s):
//   A  = strict_lower(diag(beta) (Gamma * K K^T))
//   W  = (I + A)^-1 diag(beta gamma) K,    Ut = (I + A)^-1 diag(beta) V
//   U  = Ut - W S0^T                                  (the delta-rule write vectors)
//   O  = diag(gamma) Q S0^T + lower_incl(Gamma * Q K^T) U
//   S_next = gamma_n S0 + U^T diag(exp(g_n - g)) K
// (WY representation of the gated delta rule, Yang, Kautz & Hatamizadeh, "Gated Delta
// Networks", 2024; it reaches the token recurrence's result up to rounding, which the pages
// allow for chunk boundaries: System1-Omni RFC #114, section 5.)
//
// Three launches per layer:
//   chunk_prep   (chunk, head)          : g, A, forward substitution for W and Ut   (parallel)
//   chunk_state  (sequence, head, 16 v) : U = Ut - W S^T, S <- gamma S + U^T K'     (sequential
//                                         over chunks; records each chunk's start state)
//   chunk_out    (chunk, head)          : O = gamma Q S_c^T + P U                   (parallel)
// The two small matrix products of the state pass and all of chunk_out run on the tensor
// cores (mma.sync m16n8k8 TF32 -> fp32); the state itself stays fp32.
#include <algorithm>

#include "common.cuh"

namespace s1 {
namespace gc {

constexpr int C = 64;      // chunk rows
constexpr int BV = 16;     // value rows per state-pass CTA
// D = dk = dv (64 or 128) is a template parameter of every kernel.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// Operands already rounded to TF32 when they were produced (q, k by gdn_prep; W, Ut, U and the
// recorded chunk states by the kernels below) are passed to the tensor cores as they are.
__device__ __forceinline__ uint32_t raw(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float rnd(float x) { return __uint_as_float(tf32(x)); }
// D += A(16x8, row) * B(8x8, col), tf32 inputs, fp32 accumulate
__device__ __forceinline__ void mma_tf32(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------------------
// chunk_prep: one CTA per (chunk, head), 256 threads (8 warps), two CTAs per SM.
// Writes g (within-chunk cumsum of log alpha) over loga, W and Ut (fp32 [R, H, D]).
// The unit-lower-triangular system (I + A) X = [diag(beta gamma) K | diag(beta) V] is solved
// in 16-row blocks: each 16 x 16 diagonal block's inverse comes from the nilpotent series
// (I + N)^-1 = (I - N)(I + N^2)(I + N^4)(I + N^8) (N strictly lower, N^16 = 0) in fp32, then
// X_b = T_bb (RHS_b - sum_{c<b} A_bc X_c) with the block products on the tensor cores (TF32
// in, fp32 accumulate).
template <int D>
struct PrepSmem {
  static constexpr int SX = 2 * D + 8;     // X = [K -> W | V -> Ut] ([k][n]: B(k-major) operand pattern)
  static constexpr int SA = C + 4;         // A        ([t][s]: A operand pattern)
  static constexpr int ST = 20;            // diagonal-block inverses [16][ST] (A operand pattern)
  static constexpr int SM17 = 16 * 17;     // 16 x 16 scratch matrices, row stride 17
  float X[C * SX];
  float A[C * SA];
  float T[4][16 * ST];
  float M[3][4 * SM17];                    // series scratch: N^(2^k) and products
  float g[C];
  float b[C];
};

template <int D>
__global__ void __launch_bounds__(256, 2) chunk_prep_kernel(const float* __restrict__ proj, int ld,
                                                            float* __restrict__ loga,
                                                            const float* __restrict__ beta,
                                                            const ChunkDesc* __restrict__ chunks, int H, int Dv,
                                                            float* __restrict__ Wbuf, float* __restrict__ Ubuf) {
  using SM = PrepSmem<D>;
  constexpr int SX = SM::SX, SA = SM::SA, ST = SM::ST, S17 = SM::SM17;
  constexpr int NX = 2 * D;                 // columns of X
  extern __shared__ __align__(16) uint8_t smraw[];
  SM& s = *reinterpret_cast<SM*>(smraw);
  const ChunkDesc cd = chunks[blockIdx.x];
  const int h = blockIdx.y, n = cd.len, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int HDk = H * D;
  // ---- load K (normalised) and V into X, g = cumsum(log alpha), beta
  for (int i = tid; i < C * (D / 4); i += 256) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    const bool ok = r < n;
    const float* pr = proj + (size_t)(cd.row0 + (ok ? r : 0)) * ld;
    cp16(&s.X[r * SX + c4], pr + HDk + h * D + c4, ok);
    cp16(&s.X[r * SX + D + c4], pr + 2 * HDk + h * Dv + c4, ok);
  }
  cp_commit();
  if (tid < 32) {
    const float a0 = (2 * tid < n) ? loga[(size_t)(cd.row0 + 2 * tid) * H + h] : 0.f;
    const float a1 = (2 * tid + 1 < n) ? loga[(size_t)(cd.row0 + 2 * tid + 1) * H + h] : 0.f;
    float v = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, v, o);
      if (tid >= o) v += t;
    }
    const float excl = v - (a0 + a1);
    s.g[2 * tid] = excl + a0;
    s.g[2 * tid + 1] = excl + a0 + a1;
  } else if (tid < 32 + C) {
    const int r = tid - 32;
    s.b[r] = (r < n) ? beta[(size_t)(cd.row0 + r) * H + h] : 0.f;
  }
  cp_wait<0>();
  __syncthreads();
  // ---- A = strict_lower(beta_t exp(g_t - g_s) k_t.k_s): warp -> m-tile (warp & 3), 4 n-tiles
  {
    const int r0 = (warp & 3) * 16, c0 = (warp >> 2) * 32;
    float acc[4][4] = {};
#pragma unroll 4
    for (int k = 0; k < D; k += 8) {
      const uint32_t a0 = raw(s.X[(r0 + gq) * SX + k + tq]), a1 = raw(s.X[(r0 + gq + 8) * SX + k + tq]);
      const uint32_t a2 = raw(s.X[(r0 + gq) * SX + k + tq + 4]), a3 = raw(s.X[(r0 + gq + 8) * SX + k + tq + 4]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int key = c0 + nt * 8 + gq;
        mma_tf32(acc[nt], a0, a1, a2, a3, raw(s.X[key * SX + k + tq]), raw(s.X[key * SX + k + tq + 4]));
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = r0 + gq + (e >> 1) * 8, sc = c0 + nt * 8 + 2 * tq + (e & 1);
        s.A[t * SA + sc] = (sc < t && t < n) ? rnd(s.b[t] * __expf(s.g[t] - s.g[sc]) * acc[nt][e]) : 0.f;
      }
  }
  __syncthreads();   // K rows are read by every warp above; they become the W right-hand side below
  // ---- right-hand sides in place: W half = beta_t gamma_t k_t, Ut half = beta_t v_t
  for (int i = tid; i < C * D; i += 256) {
    const int r = i / D, c = i % D;
    const float bt = s.b[r];
    s.X[r * SX + c] = rnd(s.X[r * SX + c] * (bt * __expf(s.g[r])));
    s.X[r * SX + D + c] = rnd(s.X[r * SX + D + c] * bt);
  }
  // ---- diagonal-block inverses by the nilpotent series; thread -> block bb, row i, cols j0..j0+3
  {
    const int bb = tid >> 6, e = tid & 63, i = e >> 2, j0 = (e & 3) * 4;
    float* N = s.M[0] + bb * S17;
    // N = A_bb
#pragma unroll
    for (int j = 0; j < 4; ++j) N[i * 17 + j0 + j] = s.A[(bb * 16 + i) * SA + bb * 16 + j0 + j];
    __syncthreads();
    auto mm = [&](const float* Y, const float* Z, float* o) {   // o[4] = (Y Z)[i][j0..j0+3]
      o[0] = o[1] = o[2] = o[3] = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float y = Y[i * 17 + k];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = fmaf(y, Z[k * 17 + j0 + j], o[j]);
      }
    };
    float* Pa = s.M[1] + bb * S17;
    float* Pb = s.M[2] + bb * S17;
    float o[4], tt[4];
    mm(N, N, o);                                   // P1 = N^2
#pragma unroll
    for (int j = 0; j < 4; ++j) Pa[i * 17 + j0 + j] = o[j];
    __syncthreads();
    mm(N, Pa, o);                                  // N P1
#pragma unroll
    for (int j = 0; j < 4; ++j) {                  // T1 = (I - N)(I + P1) = I - N + P1 - N P1
      const int c = j0 + j;
      tt[j] = (i == c ? 1.f : 0.f) - N[i * 17 + c] + Pa[i * 17 + c] - o[j];
    }
    mm(Pa, Pa, o);                                 // P2 = P1^2
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) { N[i * 17 + j0 + j] = tt[j]; Pb[i * 17 + j0 + j] = o[j]; }   // N <- T1
    __syncthreads();
    mm(N, Pb, o);                                  // T1 P2
#pragma unroll
    for (int j = 0; j < 4; ++j) tt[j] = N[i * 17 + j0 + j] + o[j];   // T2 = T1 (I + P2)
    mm(Pb, Pb, o);                                 // P3 = P2^2
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) { N[i * 17 + j0 + j] = tt[j]; Pa[i * 17 + j0 + j] = o[j]; }  // N <- T2
    __syncthreads();
    mm(N, Pa, o);                                  // T2 P3
#pragma unroll
    for (int j = 0; j < 4; ++j) s.T[bb][i * ST + j0 + j] = rnd(N[i * 17 + j0 + j] + o[j]);   // T3 = T2 (I + P3)
  }
  __syncthreads();
  // ---- block forward substitution over the 4 row blocks; each warp owns NT n-tiles of X
  constexpr int NT = NX / 8 / 8;           // n-tiles per warp (D=128: 4, D=64: 2)
  for (int bb = 0; bb < 4; ++bb) {
    const int r0 = bb * 16;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = (warp * NT + nt) * 8 + 2 * tq;
      acc[nt][0] = s.X[(r0 + gq) * SX + c];
      acc[nt][1] = s.X[(r0 + gq) * SX + c + 1];
      acc[nt][2] = s.X[(r0 + gq + 8) * SX + c];
      acc[nt][3] = s.X[(r0 + gq + 8) * SX + c + 1];
    }
    // R = RHS_b - A[b, 0:16b] X[0:16b]
    for (int k = 0; k < r0; k += 8) {
      const uint32_t a0 = raw(-s.A[(r0 + gq) * SA + k + tq]), a1 = raw(-s.A[(r0 + gq + 8) * SA + k + tq]);
      const uint32_t a2 = raw(-s.A[(r0 + gq) * SA + k + tq + 4]), a3 = raw(-s.A[(r0 + gq + 8) * SA + k + tq + 4]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = (warp * NT + nt) * 8 + gq;
        mma_tf32(acc[nt], a0, a1, a2, a3, raw(s.X[(k + tq) * SX + c]), raw(s.X[(k + tq + 4) * SX + c]));
      }
    }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = (warp * NT + nt) * 8 + 2 * tq;
      s.X[(r0 + gq) * SX + c] = rnd(acc[nt][0]);
      s.X[(r0 + gq) * SX + c + 1] = rnd(acc[nt][1]);
      s.X[(r0 + gq + 8) * SX + c] = rnd(acc[nt][2]);
      s.X[(r0 + gq + 8) * SX + c + 1] = rnd(acc[nt][3]);
    }
    __syncwarp();
    // X_b = T_bb R_b
    float xb[NT][4] = {};
    const float* T = s.T[bb];
#pragma unroll
    for (int k = 0; k < 16; k += 8) {
      const uint32_t a0 = raw(T[gq * ST + k + tq]), a1 = raw(T[(gq + 8) * ST + k + tq]);
      const uint32_t a2 = raw(T[gq * ST + k + tq + 4]), a3 = raw(T[(gq + 8) * ST + k + tq + 4]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int c = (warp * NT + nt) * 8 + gq;
        mma_tf32(xb[nt], a0, a1, a2, a3, raw(s.X[(r0 + k + tq) * SX + c]), raw(s.X[(r0 + k + tq + 4) * SX + c]));
      }
    }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = (warp * NT + nt) * 8 + 2 * tq;
      s.X[(r0 + gq) * SX + c] = rnd(xb[nt][0]);
      s.X[(r0 + gq) * SX + c + 1] = rnd(xb[nt][1]);
      s.X[(r0 + gq + 8) * SX + c] = rnd(xb[nt][2]);
      s.X[(r0 + gq + 8) * SX + c + 1] = rnd(xb[nt][3]);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int i = tid; i < n * (D / 4); i += 256) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    const size_t o = ((size_t)(cd.row0 + r) * H + h) * D + c4;
    *reinterpret_cast<float4*>(Wbuf + o) = *reinterpret_cast<const float4*>(&s.X[r * SX + c4]);
    *reinterpret_cast<float4*>(Ubuf + o) = *reinterpret_cast<const float4*>(&s.X[r * SX + D + c4]);
  }
  if (tid < n) loga[(size_t)(cd.row0 + tid) * H + h] = s.g[tid];
}

// ---------------------------------------------------------------------------------------
// chunk_state: one CTA per (sequence, head, block of 16 value rows), 256 threads (8 warps).
// Per chunk: U = Ut - W S^T (64 x 16, K = 128); S <- gamma_n S + U^T K' (16 x 128, K = 64),
// K'_t = exp(g_n - g_t) k_t. Records S at each chunk's start (for chunk_out) and writes U
// over Ut. The state block stays in shared memory in fp32.
template <int D, int NS>
struct StateSmem {
  static constexpr int SW = D + 4;      // W tile stride  ([t][j], A-operand pattern)
  static constexpr int SKK = D + 8;     // K tile stride  ([t][j], B-operand k-major pattern)
  static constexpr int SS = D + 4;      // state stride   ([i][j])
  static constexpr int SU = BV + 8;     // U tile stride  ([t][i])
  float W[NS][C * SW];                  // NS = 2: next chunk loads while this one computes
  float K[NS][C * SKK];
  float Ut[NS][C * BV];
  float g[NS][C];
  float S[BV * SS];
  float U[C * SU];      // U (TF32-rounded), written back for chunk_out
  float Us[C * SU];     // exp(g_n - g_t) U_t (TF32-rounded), A operand of the state update
};

// NS = 1 serves launches whose sequences have a single chunk (no prefetch needed, half the
// shared memory, two CTAs per SM). 8 warps; every matrix-product chain is split over two
// accumulators so the tensor-core latency of the sequential pass is halved.
template <int D, int NS>
__global__ void __launch_bounds__(256) chunk_state_kernel(const float* __restrict__ proj, int ld,
                                                          const float* __restrict__ gbuf,
                                                          const SeqDesc* __restrict__ seqs,
                                                          const ChunkDesc* __restrict__ chunks,
                                                          const CtxDesc* __restrict__ ctxs, int layer_g, int H,
                                                          const float* __restrict__ Wbuf, float* __restrict__ Ubuf,
                                                          float* __restrict__ Schunk, int* __restrict__ d_err) {
  extern __shared__ __align__(16) uint8_t smraw[];
  using SM = StateSmem<D, NS>;
  constexpr int SW = SM::SW, SKK = SM::SKK, SS = SM::SS, SU = SM::SU;
  constexpr int NTS = D / 64;            // 8-column n-tiles per warp in the state update
  constexpr int NTH = 256;
  SM& s = *reinterpret_cast<SM*>(smraw);
  const SeqDesc sd = seqs[blockIdx.x];
  const int h = blockIdx.y, v0 = blockIdx.z * BV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int HDk = H * D;
  const size_t head_off = (size_t)(layer_g * H + h) * D * D;
  const float* S0 = sd.ctx_in >= 0 ? ctxs[sd.ctx_in].S + head_off : nullptr;
  for (int i = tid; i < BV * D; i += NTH) {
    const int r = i / D, c = i % D;
    s.S[r * SS + c] = S0 ? S0[(size_t)(v0 + r) * D + c] : 0.f;
  }
  const int nch = (sd.len + C - 1) / C;
  auto load = [&](int cl, int st) {
    const ChunkDesc cd = chunks[sd.chunk0 + cl];
    for (int i = tid; i < C * (D / 4); i += NTH) {
      const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
      const bool okr = r < cd.len;
      const int row = cd.row0 + (okr ? r : 0);
      cp16(&s.W[st][r * SW + c4], Wbuf + ((size_t)row * H + h) * D + c4, okr);
      cp16(&s.K[st][r * SKK + c4], proj + (size_t)row * ld + HDk + h * D + c4, okr);
    }
    for (int i = tid; i < C * (BV / 4); i += NTH) {
      const int r = i / (BV / 4), c4 = (i % (BV / 4)) * 4;
      const bool okr = r < cd.len;
      const int row = cd.row0 + (okr ? r : 0);
      cp16(&s.Ut[st][r * BV + c4], Ubuf + ((size_t)row * H + h) * D + v0 + c4, okr);
    }
    if (tid < C) s.g[st][tid] = tid < cd.len ? gbuf[(size_t)(cd.row0 + tid) * H + h] : 0.f;
  };
  if (nch > 0) load(0, 0);
  cp_commit();
  const bool ok = true;
  for (int cl = 0; cl < nch; ++cl) {
    const int st = NS == 2 ? (cl & 1) : 0;
    const ChunkDesc cd = chunks[sd.chunk0 + cl];
    if (NS == 2) {
      if (cl + 1 < nch) load(cl + 1, st ^ 1);
      cp_commit();
      cp_wait<1>();
    } else {
      if (cl > 0) load(cl, 0);   // single stage: the previous chunk's tiles are no longer read
      cp_commit();
      cp_wait<0>();
    }
    __syncthreads();
    // record the chunk-start state block
    {
      float* dst = Schunk + ((size_t)(sd.chunk0 + cl) * H + h) * D * D + (size_t)v0 * D;
      for (int i = tid; i < BV * (D / 4); i += NTH) {
        const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
        const float4 v = *reinterpret_cast<const float4*>(&s.S[r * SS + c4]);
        *reinterpret_cast<float4*>(dst + (size_t)r * D + c4) = make_float4(rnd(v.x), rnd(v.y), rnd(v.z), rnd(v.w));
      }
    }
    // U = Ut - W S^T : warp -> rows 16*(warp&3) .., value columns 8*(warp>>2) .. +7
    {
      float a0c[4] = {0.f, 0.f, 0.f, 0.f}, a1c[4] = {0.f, 0.f, 0.f, 0.f};
      const float* Wt = s.W[st];
      const int r0 = (warp & 3) * 16, n0 = (warp >> 2) * 8;
#pragma unroll 4
      for (int k = 0; k < D; k += 16) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int kk = k + half * 8;
          const uint32_t x0 = raw(Wt[(r0 + gq) * SW + kk + tq]), x1 = raw(Wt[(r0 + gq + 8) * SW + kk + tq]);
          const uint32_t x2 = raw(Wt[(r0 + gq) * SW + kk + tq + 4]), x3 = raw(Wt[(r0 + gq + 8) * SW + kk + tq + 4]);
          const uint32_t b0 = tf32(s.S[(n0 + gq) * SS + kk + tq]), b1 = tf32(s.S[(n0 + gq) * SS + kk + tq + 4]);
          mma_tf32(half ? a1c : a0c, x0, x1, x2, x3, b0, b1);
        }
      }
      const int c = n0 + 2 * tq;
      const int ra = r0 + gq, rb = r0 + gq + 8;
      const float gn = s.g[st][cd.len - 1];
      const float ea = __expf(gn - s.g[st][ra]), eb = __expf(gn - s.g[st][rb]);
      const float u0 = s.Ut[st][ra * BV + c] - (a0c[0] + a1c[0]), u1 = s.Ut[st][ra * BV + c + 1] - (a0c[1] + a1c[1]);
      const float u2 = s.Ut[st][rb * BV + c] - (a0c[2] + a1c[2]), u3 = s.Ut[st][rb * BV + c + 1] - (a0c[3] + a1c[3]);
      s.U[ra * SU + c] = rnd(u0);
      s.U[ra * SU + c + 1] = rnd(u1);
      s.U[rb * SU + c] = rnd(u2);
      s.U[rb * SU + c + 1] = rnd(u3);
      s.Us[ra * SU + c] = rnd(ea * u0);
      s.Us[ra * SU + c + 1] = rnd(ea * u1);
      s.Us[rb * SU + c] = rnd(eb * u2);
      s.Us[rb * SU + c + 1] = rnd(eb * u3);
    }
    __syncthreads();
    // write U (this block's 16 value columns) over Ut
    for (int i = tid; i < cd.len * (BV / 4); i += NTH) {
      const int r = i / (BV / 4), c4 = (i % (BV / 4)) * 4;
      *reinterpret_cast<float4*>(Ubuf + ((size_t)(cd.row0 + r) * H + h) * D + v0 + c4) =
          make_float4(s.U[r * SU + c4], s.U[r * SU + c4 + 1], s.U[r * SU + c4 + 2], s.U[r * SU + c4 + 3]);
    }
    // S <- gamma_n S + U^T K' : warp -> value rows 0..15, key columns 8*NTS*warp .. (NTS n-tiles)
    // (not needed after the last chunk of a sequence whose final state nobody keeps)
    if (cl + 1 < nch || sd.ctx_out >= 0) {
      const float gn = s.g[st][cd.len - 1];
      const float gam = __expf(gn);
      float acc[NTS][4], acc2[NTS][4];
#pragma unroll
      for (int nt = 0; nt < NTS; ++nt) {
        const int c = warp * (8 * NTS) + nt * 8 + 2 * tq;
        acc[nt][0] = gam * s.S[gq * SS + c];
        acc[nt][1] = gam * s.S[gq * SS + c + 1];
        acc[nt][2] = gam * s.S[(gq + 8) * SS + c];
        acc[nt][3] = gam * s.S[(gq + 8) * SS + c + 1];
        acc2[nt][0] = acc2[nt][1] = acc2[nt][2] = acc2[nt][3] = 0.f;
      }
      const float* Kt = s.K[st];
#pragma unroll 2
      for (int k = 0; k < C; k += 16) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int kk = k + half * 8;
          // A[i][t] = exp(g_n - g_t) U[t][i]
          const uint32_t x0 = raw(s.Us[(kk + tq) * SU + gq]), x1 = raw(s.Us[(kk + tq) * SU + gq + 8]);
          const uint32_t x2 = raw(s.Us[(kk + tq + 4) * SU + gq]), x3 = raw(s.Us[(kk + tq + 4) * SU + gq + 8]);
#pragma unroll
          for (int nt = 0; nt < NTS; ++nt) {
            const int c = warp * (8 * NTS) + nt * 8 + gq;
            mma_tf32(half ? acc2[nt] : acc[nt], x0, x1, x2, x3, raw(Kt[(kk + tq) * SKK + c]),
                     raw(Kt[(kk + tq + 4) * SKK + c]));
          }
        }
      }
      __syncthreads();   // every warp has read S and U
#pragma unroll
      for (int nt = 0; nt < NTS; ++nt) {
        const int c = warp * (8 * NTS) + nt * 8 + 2 * tq;
        s.S[gq * SS + c] = acc[nt][0] + acc2[nt][0];
        s.S[gq * SS + c + 1] = acc[nt][1] + acc2[nt][1];
        s.S[(gq + 8) * SS + c] = acc[nt][2] + acc2[nt][2];
        s.S[(gq + 8) * SS + c + 1] = acc[nt][3] + acc2[nt][3];
      }
    }
    __syncthreads();
  }
  if (ok && sd.ctx_out >= 0) {
    float* So = ctxs[sd.ctx_out].S + head_off;
    for (int i = tid; i < BV * D; i += NTH) {
      const int r = i / D, c = i % D;
      So[(size_t)(v0 + r) * D + c] = s.S[r * SS + c];
    }
  }
}

// ---------------------------------------------------------------------------------------
// chunk_out: one CTA per (chunk, head), 256 threads (8 warps).
// O = diag(gamma) Q S_c^T + P U, P = lower_incl(Gamma * Q K^T); out bf16 [R, H*Dv].
template <int D>
struct OutSmem {
  static constexpr int SQ = D + 4;   // Q, K tiles ([t][j], A / B(n-major) pattern)
  static constexpr int SSC = D + 4;  // chunk-start state ([i][j])
  static constexpr int SUo = D + 8;  // U tile ([s][i], B k-major pattern)
  static constexpr int SP = C + 4;   // P ([t][s])
  float Q[C * SQ];
  float KU[C * SUo];        // K, then U
  float S[D * SSC];
  float P[C * SP];
  float g[C];
};

template <int D>
__global__ void __launch_bounds__(256) chunk_out_kernel(const float* __restrict__ proj, int ld,
                                                        const float* __restrict__ gbuf,
                                                        const ChunkDesc* __restrict__ chunks, int H,
                                                        const float* __restrict__ Ubuf,
                                                        const float* __restrict__ Schunk, bf16* __restrict__ out) {
  allow_dependents();
  extern __shared__ __align__(16) uint8_t smraw[];
  using SM = OutSmem<D>;
  constexpr int SQ = SM::SQ, SSC = SM::SSC, SUo = SM::SUo, SP = SM::SP;
  constexpr int NTO = D / 16;            // 8-column n-tiles per warp of the output
  SM& s = *reinterpret_cast<SM*>(smraw);
  const int ci = blockIdx.x, h = blockIdx.y;
  const ChunkDesc cd = chunks[ci];
  const int n = cd.len;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int HDk = H * D;
  for (int i = tid; i < C * (D / 4); i += 256) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    const bool ok = r < n;
    const int row = cd.row0 + (ok ? r : 0);
    cp16(&s.Q[r * SQ + c4], proj + (size_t)row * ld + h * D + c4, ok);
    cp16(&s.KU[r * SQ + c4], proj + (size_t)row * ld + HDk + h * D + c4, ok);   // K with the Q stride
  }
  const float* Sc = Schunk + ((size_t)ci * H + h) * D * D;
  for (int i = tid; i < D * (D / 4); i += 256) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    cp16(&s.S[r * SSC + c4], Sc + (size_t)r * D + c4, true);
  }
  if (tid < C) s.g[tid] = tid < n ? gbuf[(size_t)(cd.row0 + tid) * H + h] : 0.f;
  cp_commit();
  cp_wait<0>();
  __syncthreads();
  const int mt = warp & 3;          // 16-row m-tile
  const int r0 = mt * 16;
  // P = lower_incl(exp(g_t - g_s) q_t.k_s): warp -> rows r0.., key columns 32*(warp>>2) .. +31
  {
    float acc[4][4] = {};
    const int c0 = (warp >> 2) * 32;
#pragma unroll 4
    for (int k = 0; k < D; k += 8) {
      const uint32_t a0 = raw(s.Q[(r0 + gq) * SQ + k + tq]), a1 = raw(s.Q[(r0 + gq + 8) * SQ + k + tq]);
      const uint32_t a2 = raw(s.Q[(r0 + gq) * SQ + k + tq + 4]), a3 = raw(s.Q[(r0 + gq + 8) * SQ + k + tq + 4]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int key = c0 + nt * 8 + gq;
        const uint32_t b0 = raw(s.KU[key * SQ + k + tq]), b1 = raw(s.KU[key * SQ + k + tq + 4]);
        mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = r0 + gq + (e >> 1) * 8, sidx = c0 + nt * 8 + 2 * tq + (e & 1);
        s.P[t * SP + sidx] = (sidx <= t && t < n) ? rnd(__expf(s.g[t] - s.g[sidx]) * acc[nt][e]) : 0.f;
      }
    }
  }
  __syncthreads();
  // U tile over K (k-major stride)
  for (int i = tid; i < C * (D / 4); i += 256) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    const bool ok = r < n;
    const int row = cd.row0 + (ok ? r : 0);
    cp16(&s.KU[r * SUo + c4], Ubuf + ((size_t)row * H + h) * D + c4, ok);
  }
  cp_commit();
  // O1 = Q S_c^T  (warp -> rows r0.., value columns (D/2)*(warp>>2) .. : NTO n-tiles)
  float o[NTO][4] = {};
  const int cbase = (warp >> 2) * (D / 2);
#pragma unroll 2
  for (int k = 0; k < D; k += 8) {
    const uint32_t a0 = raw(s.Q[(r0 + gq) * SQ + k + tq]), a1 = raw(s.Q[(r0 + gq + 8) * SQ + k + tq]);
    const uint32_t a2 = raw(s.Q[(r0 + gq) * SQ + k + tq + 4]), a3 = raw(s.Q[(r0 + gq + 8) * SQ + k + tq + 4]);
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      const int i = cbase + nt * 8 + gq;
      const uint32_t b0 = raw(s.S[i * SSC + k + tq]), b1 = raw(s.S[i * SSC + k + tq + 4]);
      mma_tf32(o[nt], a0, a1, a2, a3, b0, b1);
    }
  }
  {
    const float ga = __expf(s.g[r0 + gq]), gb = __expf(s.g[r0 + gq + 8]);
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) { o[nt][0] *= ga; o[nt][1] *= ga; o[nt][2] *= gb; o[nt][3] *= gb; }
  }
  cp_wait<0>();
  __syncthreads();
  // O += P U
#pragma unroll 2
  for (int k = 0; k < C; k += 8) {
    const uint32_t a0 = raw(s.P[(r0 + gq) * SP + k + tq]), a1 = raw(s.P[(r0 + gq + 8) * SP + k + tq]);
    const uint32_t a2 = raw(s.P[(r0 + gq) * SP + k + tq + 4]), a3 = raw(s.P[(r0 + gq + 8) * SP + k + tq + 4]);
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      const int i = cbase + nt * 8 + gq;
      const uint32_t b0 = raw(s.KU[(k + tq) * SUo + i]), b1 = raw(s.KU[(k + tq + 4) * SUo + i]);
      mma_tf32(o[nt], a0, a1, a2, a3, b0, b1);
    }
  }
  const int HDv = H * D;
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) {
    const int c = cbase + nt * 8 + 2 * tq;
    const int ta = r0 + gq, tb = r0 + gq + 8;
    if (ta < n)
      *reinterpret_cast<__nv_bfloat162*>(out + (size_t)(cd.row0 + ta) * HDv + h * D + c) =
          __floats2bfloat162_rn(o[nt][0], o[nt][1]);
    if (tb < n)
      *reinterpret_cast<__nv_bfloat162*>(out + (size_t)(cd.row0 + tb) * HDv + h * D + c) =
          __floats2bfloat162_rn(o[nt][2], o[nt][3]);
  }
}

}  // namespace gc

bool gdn_chunked_supported(int H, int Dk, int Dv, int ld) {
  return Dk == Dv && (Dk == 64 || Dk == 128) && H > 0 && (ld % 4) == 0;
}

template <int D>
static cudaError_t launch_state(const float* proj, int ld, const float* g, const SeqDesc* d_seq, int n_seq,
                                const ChunkDesc* d_chunks, const CtxDesc* d_ctx, int layer_g, int H,
                                const float* Wbuf, float* Ubuf, float* Schunk, int max_chunks, int* d_err,
                                cudaStream_t st) {
  if (n_seq <= 0) return cudaSuccess;
  const dim3 grid(n_seq, H, D / gc::BV);
  if (max_chunks <= 1) {
    gc::chunk_state_kernel<D, 1><<<grid, 256, sizeof(gc::StateSmem<D, 1>), st>>>(
        proj, ld, g, d_seq, d_chunks, d_ctx, layer_g, H, Wbuf, Ubuf, Schunk, d_err);
  } else {
    gc::chunk_state_kernel<D, 2><<<grid, 256, sizeof(gc::StateSmem<D, 2>), st>>>(
        proj, ld, g, d_seq, d_chunks, d_ctx, layer_g, H, Wbuf, Ubuf, Schunk, d_err);
  }
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_chunked_d(float* proj, int ld, float* loga, const float* beta, bf16* out,
                                    const SeqDesc* d_seq, int n_seq, const ChunkDesc* d_chunks, int n_chunks,
                                    const CtxDesc* d_ctx, int layer_g, int H, float* Wbuf, float* Ubuf,
                                    float* Schunk, int n_first, int max_chunks_first, int max_chunks_rest,
                                    int* d_err, cudaStream_t st) {
  static bool attr = false;
  const size_t sp = sizeof(gc::PrepSmem<D>);
  const size_t so = sizeof(gc::OutSmem<D>);
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gc::chunk_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_state_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(gc::StateSmem<D, 1>));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_state_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(gc::StateSmem<D, 2>));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_out_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)so);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  gc::chunk_prep_kernel<D><<<dim3(n_chunks, H), 256, sp, st>>>(proj, ld, loga, beta, d_chunks, H, D, Wbuf, Ubuf);
  // sequences [0, n_first) run before the rest (the rest continue from their states)
  const int split = (n_first > 0 && n_first < n_seq) ? n_first : n_seq;
  cudaError_t e = launch_state<D>(proj, ld, loga, d_seq, split, d_chunks, d_ctx, layer_g, H, Wbuf, Ubuf, Schunk,
                                  split < n_seq ? max_chunks_first : std::max(max_chunks_first, max_chunks_rest),
                                  d_err, st);
  if (e != cudaSuccess) return e;
  if (split < n_seq) {
    e = launch_state<D>(proj, ld, loga, d_seq + split, n_seq - split, d_chunks, d_ctx, layer_g, H, Wbuf, Ubuf,
                        Schunk, max_chunks_rest, d_err, st);
    if (e != cudaSuccess) return e;
  }
  gc::chunk_out_kernel<D><<<dim3(n_chunks, H), 256, so, st>>>(proj, ld, loga, d_chunks, H, Ubuf, Schunk, out);
  return cudaGetLastError();
}

cudaError_t launch_gdn_chunked(float* proj, int ld, float* loga, const float* beta, bf16* out,
                               const SeqDesc* d_seq, int n_seq, const ChunkDesc* d_chunks, int n_chunks,
                               const CtxDesc* d_ctx, int layer_g, int H, int Dk, int Dv, float* Wbuf, float* Ubuf,
                               float* Schunk, int n_first, int max_chunks_first, int max_chunks_rest,
                               int* d_err, cudaStream_t st, long* launches) {
  if (n_seq <= 0 || n_chunks <= 0) return cudaSuccess;
  if (!gdn_chunked_supported(H, Dk, Dv, ld)) return cudaErrorNotSupported;
  if (n_seq > 65535 || n_chunks > 2147483647 / 2) return cudaErrorInvalidValue;
  cudaError_t e = (Dk == 128)
                      ? launch_chunked_d<128>(proj, ld, loga, beta, out, d_seq, n_seq, d_chunks, n_chunks, d_ctx,
                                              layer_g, H, Wbuf, Ubuf, Schunk, n_first, max_chunks_first,
                                              max_chunks_rest, d_err, st)
                      : launch_chunked_d<64>(proj, ld, loga, beta, out, d_seq, n_seq, d_chunks, n_chunks, d_ctx,
                                             layer_g, H, Wbuf, Ubuf, Schunk, n_first, max_chunks_first,
                                             max_chunks_rest, d_err, st);
  if (launches) *launches += (n_first > 0 && n_first < n_seq) ? 4 : 3;
  return e;
}

}  // namespace s1
