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
// Launches per layer (the gated delta rule's gates and q/k L2 norms are formed inside them):
//   chunk_prep   (chunk, head)          : gates, k norm, g, A, forward substitution for W, Ut
//                                         (parallel)
//   chunk_state  (sequence, head, 16 v) : U = Ut - W S^T, S <- gamma S + U^T K'     (sequential
//                                         over chunks; records each chunk's start state)
//   chunk_out    (chunk, head)          : q norm, O = gamma Q S_c^T + P U           (parallel)
// Single-chunk sequences that keep no state need no state pass: in a one-sweep call the
// prefix's pass also serves the questions that continue from it; otherwise chunk_out forms
// their U from the start state itself. The small matrix products run on the tensor cores
// (mma.sync m16n8k8 TF32 -> fp32); the state itself stays fp32.
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
// Operands already rounded to TF32 when they were produced (k by chunk_prep, q by chunk_out;
// W, Ut, U and the recorded chunk states by the kernels below) go to the tensor cores as they are.
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
  float la[C];                             // log alpha
};

template <int D>
__global__ void __launch_bounds__(256, 2) chunk_prep_kernel(float* __restrict__ proj, int ld,
                                                            float* __restrict__ loga,
                                                            const ChunkDesc* __restrict__ chunks, int H, int Dv,
                                                            float eps, float* __restrict__ Wbuf,
                                                            float* __restrict__ Ubuf) {
  allow_dependents();
  wait_prerequisites();
  using SM = PrepSmem<D>;
  constexpr int SX = SM::SX, SA = SM::SA, ST = SM::ST, S17 = SM::SM17;
  constexpr int NX = 2 * D;                 // columns of X
  extern __shared__ __align__(16) uint8_t smraw[];
  SM& s = *reinterpret_cast<SM*>(smraw);
  const ChunkDesc cd = chunks[blockIdx.x];
  const int h = blockIdx.y, n = cd.len, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int HDk = H * D;
  // ---- load K and V into X; gates from the a, b columns of the projection
  for (int i = tid; i < C * (D / 4); i += 256) {
    const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
    const bool ok = r < n;
    const float* pr = proj + (size_t)(cd.row0 + (ok ? r : 0)) * ld;
    cp16(&s.X[r * SX + c4], pr + HDk + h * D + c4, ok);
    cp16(&s.X[r * SX + D + c4], pr + 2 * HDk + h * Dv + c4, ok);
  }
  cp_commit();
  if (tid < C) {
    // alpha_t = exp(-softplus(a_t)), beta_t = sigmoid(b_t)
    float la = 0.f, bt = 0.f;
    if (tid < n) {
      const float* ab = proj + (size_t)(cd.row0 + tid) * ld + 2 * HDk + H * Dv;
      const float a = ab[h], b = ab[H + h];
      la = -(fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))));
      bt = 1.f / (1.f + expf(-b));
    }
    s.la[tid] = la;
    s.b[tid] = bt;
  }
  cp_wait<0>();
  __syncthreads();
  // g = cumsum(log alpha) within the chunk (one warp, two rows per lane)
  if (tid < 32) {
    const float a0 = s.la[2 * tid], a1 = s.la[2 * tid + 1];
    float v = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, v, o);
      if (tid >= o) v += t;
    }
    const float excl = v - (a0 + a1);
    s.g[2 * tid] = excl + a0;
    s.g[2 * tid + 1] = excl + a0 + a1;
  }
  // k <- k / sqrt(sum k^2 + eps), rounded to TF32 (every later product of k runs on TF32 tensor-core
  // inputs), in shared memory and back in the projection for the later kernels; four threads per
  // row. (q is normalised the same way where it is used, in chunk_out.)
  {
    constexpr int PER = D / 4;
    const int r = tid >> 2, sub = tid & 3;
    float* xs = &s.X[r * SX + sub * PER];
    float v[PER];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
      const float4 t = *reinterpret_cast<const float4*>(xs + i);
      v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) ss += v[i] * v[i];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = 1.0f / sqrtf(ss + eps);
    if (r < n) {
      float* kg = proj + (size_t)(cd.row0 + r) * ld + HDk + h * D + sub * PER;
#pragma unroll
      for (int i = 0; i < PER; i += 4) {
        const float4 t = make_float4(rnd(v[i] * inv), rnd(v[i + 1] * inv), rnd(v[i + 2] * inv), rnd(v[i + 3] * inv));
        *reinterpret_cast<float4*>(xs + i) = t;
        *reinterpret_cast<float4*>(kg + i) = t;
      }
    }
  }
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
// chunk_state: one CTA per (sequence, head, block of 16 value rows), 512 threads (16 warps).
// Per chunk: U = Ut - W S^T (64 x 16, K = D); S <- gamma_n S + U^T K' (16 x D, K = 64),
// K'_t = exp(g_n - g_t) k_t. Records each chunk's start state (TF32-rounded, for chunk_out)
// and writes U over Ut. The state block stays in shared memory in fp32, next to a TF32-rounded
// copy that feeds the tensor cores.
//
// The chunk tiles W, K (64 x D fp32) and Ut (64 x 16) arrive by TMA, issued by one thread one
// chunk ahead, into 128-byte-swizzled boxes of 32 columns: ldmatrix then reads conflict-free
// 8-row fragments (a TF32 fragment row is four 32-bit values = one 16-byte ldmatrix row).
// Rows of a partial chunk past its end hold the following rows of the buffers (or zeros past
// the last row); they only ever meet zero coefficients (Us rows past the end are set to 0).
template <int D, int NS>
struct StateSmem {
  static constexpr int NB = D / 32;     // 32-column boxes per tile row
  static constexpr int SS = D + 4;      // fp32 state stride ([i][j])
  static constexpr int SU = BV + 8;     // U stride ([t][i])
  static constexpr int SUT = C + 4;     // Us^T stride ([i][t], ldmatrix rows 16-byte aligned)
  float W[NS][C * D];                   // NB boxes [64][32], swizzled
  float K[NS][C * D];
  float Sr[BV * D];                     // TF32-rounded state, NB boxes [16][32], swizzled
  float Ut[NS][C * BV];                 // [64][16] dense
  float S[BV * SS];
  float U[C * SU];                      // U (TF32-rounded), written back for chunk_out
  float UsT[BV * SUT];                  // exp(g_n - g_t) U_t, transposed (TF32-rounded)
  float Up[C * BV];                     // second key half's partial W S^T
  float g[NS][C];
  uint64_t full[NS];
};

// float index of (row, col) in a 128-byte-swizzled box of 32 fp32 columns
__device__ __forceinline__ int swz32(int row, int col) {
  return row * 32 + ((((col >> 2) ^ (row & 7))) << 2) + (col & 3);
}
__device__ __forceinline__ void ldsm4(const float* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void cp4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (about 1 s of %globaltimer); false on expiry.
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
  if (bar_try(bar, parity)) return true;
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t it = 1;; ++it) {
    if (bar_try(bar, parity)) return true;
    if ((it & 255) == 0) {
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 1000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void tma2(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tma_store2(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Maps: mapW over Wbuf [R, H, D] (box 32 x 1 x 64, swizzled), mapUt over Ubuf [R, H, D] (box
// 16 x 1 x 64, dense), mapK over proj [R, ld] (box 32 x 64, swizzled), mapSc over the chunk-start
// records [n_chunks * H * D, D] (box 32 x 16, swizzled like Sr).
// NS = 1 serves launches whose sequences have a single chunk (half the shared memory, two CTAs
// per SM).
template <int D, int NS>
__global__ void __launch_bounds__(512) chunk_state_kernel(const __grid_constant__ CUtensorMap mapW,
                                                          const __grid_constant__ CUtensorMap mapK,
                                                          const __grid_constant__ CUtensorMap mapUt,
                                                          const __grid_constant__ CUtensorMap mapSc,
                                                          const float* __restrict__ gbuf,
                                                          const SeqDesc* __restrict__ seqs,
                                                          const ChunkDesc* __restrict__ chunks,
                                                          const CtxDesc* __restrict__ ctxs, int layer_g, int H,
                                                          float* __restrict__ Ubuf, float* __restrict__ Schunk,
                                                          int* __restrict__ d_err) {
  allow_dependents();
  wait_prerequisites();
  extern __shared__ __align__(16) uint8_t smraw[];   // (rounded up to 1024 bytes below)
  using SM = StateSmem<D, NS>;
  constexpr int SS = SM::SS, SU = SM::SU, SUT = SM::SUT, NB = SM::NB;
  constexpr int NTH = 512;               // 16 warps
  constexpr int NUPD = D / 8;            // warps of the state update (one 8-column n-tile each)
  constexpr uint32_t TILE_BYTES = 2 * C * D * 4 + C * BV * 4;
  SM& s = *reinterpret_cast<SM*>((((uintptr_t)smraw) + 1023) & ~(uintptr_t)1023);
  const SeqDesc sd = seqs[blockIdx.x];
  const int h = blockIdx.y, v0 = blockIdx.z * BV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int HDk = H * D;
  const int nch = (sd.len + C - 1) / C;
  // followers: single-chunk sequences continuing from this one's final state; each adds one
  // step after the last chunk (U and the chunk-start record from the final state, no update)
  const int nf = sd.fol1 > sd.fol0 ? sd.fol1 - sd.fol0 : 0;
  const int nsteps = nch + nf;
  auto chunk_of = [&](int cl) { return cl < nch ? sd.chunk0 + cl : seqs[sd.fol0 + (cl - nch)].chunk0; };
  const size_t head_off = (size_t)(layer_g * H + h) * D * D;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) bar_init(&s.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // step descriptors (chunk index + chunk) are fetched two steps ahead, so no step waits on a
  // global load before issuing its TMA or using its row range
  struct Step { int ci; ChunkDesc cd; };
  auto fetch = [&](int cl) -> Step {
    if (cl >= nsteps) return Step{0, ChunkDesc{0, 1, 0}};
    const int ci = chunk_of(cl);
    return Step{ci, chunks[ci]};
  };
  auto issue = [&](const ChunkDesc& cd, int st) {   // one thread: TMA of a step's tiles into stage st
    bar_expect_tx(&s.full[st], TILE_BYTES);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      tma3(&s.W[st][b * C * 32], &mapW, &s.full[st], 32 * b, h, cd.row0);
      tma2(&s.K[st][b * C * 32], &mapK, &s.full[st], HDk + h * D + 32 * b, cd.row0);
    }
    tma3(&s.Ut[st][0], &mapUt, &s.full[st], v0, h, cd.row0);
  };
  auto load_g = [&](const ChunkDesc& cd, int st) {
    if (tid < C) cp4(&s.g[st][tid], gbuf + (size_t)(cd.row0 + (tid < cd.len ? tid : 0)) * H + h, tid < cd.len);
  };
  Step s0 = fetch(0), s1 = fetch(1);
  if (nsteps > 0 && tid == 0) issue(s0.cd, 0);
  if (nsteps > 0) load_g(s0.cd, 0);
  cp_commit();
  // initial state block: fp32 and TF32-rounded copies
  const float* S0 = sd.ctx_in >= 0 ? ctxs[sd.ctx_in].S + head_off : nullptr;
  for (int i = tid; i < BV * D; i += NTH) {
    const int r = i / D, c = i % D;
    const float v = S0 ? S0[(size_t)(v0 + r) * D + c] : 0.f;
    s.S[r * SS + c] = v;
    s.Sr[(c >> 5) * (BV * 32) + swz32(r, c & 31)] = rnd(v);
  }
  fence_async_smem();   // Sr is read by bulk stores
  bool ok = true;
  for (int cl = 0; cl < nsteps; ++cl) {
    const int st = NS == 2 ? (cl & 1) : 0;
    const Step s2 = fetch(cl + 2);   // used two steps from now
    const int ci = s0.ci;
    const ChunkDesc cd = s0.cd;
    if (NS == 2) {
      if (cl + 1 < nsteps) {
        if (tid == 0) issue(s1.cd, st ^ 1);
        load_g(s1.cd, st ^ 1);
      }
      cp_commit();
      cp_wait<1>();
    } else {
      if (cl > 0) {   // single stage: the previous chunk's tiles are no longer read
        if (tid == 0) issue(cd, 0);
        load_g(cd, 0);
      }
      cp_commit();
      cp_wait<0>();
    }
    s0 = s1;
    s1 = s2;
    // every thread waits (bounded) for the chunk's tiles; one barrier agrees on the outcome, so
    // all threads take the same path
    const uint32_t parity = NS == 2 ? ((cl >> 1) & 1) : (cl & 1);
    if (!__syncthreads_and(bar_wait(&s.full[st], parity) ? 1 : 0)) {
      if (tid == 0) atomicExch(d_err, 0x201);
      ok = false;
      break;
    }
    // record the chunk-start state block (already rounded, in the map's swizzled box layout) for
    // chunk_out: one bulk store per 32-column box, read asynchronously from Sr
    if (tid == 0) {
      fence_async_smem();
      const int y = (ci * H + h) * D + v0;
#pragma unroll
      for (int b = 0; b < NB; ++b) tma_store2(&mapSc, &s.Sr[b * (BV * 32)], 32 * b, y);
      bulk_commit();
    }
    // U = Ut - W S^T : warp -> rows 16*(warp&3) .., value columns 8*((warp>>2)&1) .. +7, key
    // half (warp>>3) of the contraction; the two halves meet in shared memory
    {
      float a0c[4] = {0.f, 0.f, 0.f, 0.f}, a1c[4] = {0.f, 0.f, 0.f, 0.f};
      const float* Wt = s.W[st];
      const int r0 = (warp & 3) * 16, n0 = ((warp >> 2) & 1) * 8, kh = warp >> 3;
      const int mi = lane >> 3;
      const int arow = r0 + (lane & 7) + 8 * (mi & 1), acol = 4 * (mi >> 1);   // A: ldmatrix lane row
      const int brow = n0 + (lane & 7), bcol = 4 * mi;                          // B: ldmatrix lane row
#pragma unroll
      for (int k = kh * (D / 2); k < (kh + 1) * (D / 2); k += 16) {
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3, b0, b1, b2, b3;
        {
          const int c = k + acol;
          ldsm4(&Wt[(c >> 5) * (C * 32) + swz32(arow, c & 31)], x0, x1, x2, x3);
          const int c2 = k + 8 + acol;
          ldsm4(&Wt[(c2 >> 5) * (C * 32) + swz32(arow, c2 & 31)], y0, y1, y2, y3);
          const int cb = k + bcol;
          ldsm4(&s.Sr[(cb >> 5) * (BV * 32) + swz32(brow, cb & 31)], b0, b1, b2, b3);
        }
        mma_tf32(a0c, x0, x1, x2, x3, b0, b1);
        mma_tf32(a1c, y0, y1, y2, y3, b2, b3);
      }
      const int c = n0 + 2 * tq;
      const int ra = r0 + gq, rb = r0 + gq + 8;
      if (kh == 1) {
        s.Up[ra * BV + c] = a0c[0] + a1c[0];
        s.Up[ra * BV + c + 1] = a0c[1] + a1c[1];
        s.Up[rb * BV + c] = a0c[2] + a1c[2];
        s.Up[rb * BV + c + 1] = a0c[3] + a1c[3];
      }
      __syncthreads();
      if (kh == 0) {
        const float gn = s.g[st][cd.len - 1];
        const float ea = __expf(gn - s.g[st][ra]), eb = __expf(gn - s.g[st][rb]);
        const float u0 = s.Ut[st][ra * BV + c] - ((a0c[0] + a1c[0]) + s.Up[ra * BV + c]);
        const float u1 = s.Ut[st][ra * BV + c + 1] - ((a0c[1] + a1c[1]) + s.Up[ra * BV + c + 1]);
        const float u2 = s.Ut[st][rb * BV + c] - ((a0c[2] + a1c[2]) + s.Up[rb * BV + c]);
        const float u3 = s.Ut[st][rb * BV + c + 1] - ((a0c[3] + a1c[3]) + s.Up[rb * BV + c + 1]);
        s.U[ra * SU + c] = rnd(u0);
        s.U[ra * SU + c + 1] = rnd(u1);
        s.U[rb * SU + c] = rnd(u2);
        s.U[rb * SU + c + 1] = rnd(u3);
        const bool oka = ra < cd.len, okb = rb < cd.len;
        s.UsT[c * SUT + ra] = oka ? rnd(ea * u0) : 0.f;
        s.UsT[(c + 1) * SUT + ra] = oka ? rnd(ea * u1) : 0.f;
        s.UsT[c * SUT + rb] = okb ? rnd(eb * u2) : 0.f;
        s.UsT[(c + 1) * SUT + rb] = okb ? rnd(eb * u3) : 0.f;
      }
    }
    __syncthreads();
    // write U (this block's 16 value columns) over Ut
    for (int i = tid; i < cd.len * (BV / 4); i += NTH) {
      const int r = i / (BV / 4), c4 = (i % (BV / 4)) * 4;
      *reinterpret_cast<float4*>(Ubuf + ((size_t)(cd.row0 + r) * H + h) * D + v0 + c4) =
          make_float4(s.U[r * SU + c4], s.U[r * SU + c4 + 1], s.U[r * SU + c4 + 2], s.U[r * SU + c4 + 3]);
    }
    // S <- gamma_n S + Us^T K : warp w < D/8 -> value rows 0..15, key columns 8w .. 8w+7
    // (not needed after the last chunk of a sequence whose final state nobody keeps, nor for
    // followers)
    if (cl < nch && (cl + 1 < nch || sd.ctx_out >= 0)) {
      const float gam = __expf(s.g[st][cd.len - 1]);
      const bool upd = warp < NUPD;
      const int c = warp * 8 + 2 * tq;   // this lane's output columns c, c+1 (warp's n-tile)
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
      if (upd) {
        acc[0] = gam * s.S[gq * SS + c];
        acc[1] = gam * s.S[gq * SS + c + 1];
        acc[2] = gam * s.S[(gq + 8) * SS + c];
        acc[3] = gam * s.S[(gq + 8) * SS + c + 1];
        const float* Kt = s.K[st];
        const int mi = lane >> 3;
        const int arow = (lane & 7) + 8 * (mi & 1), acol = 4 * (mi >> 1);
        const int j = warp * 8 + gq;
        const float* kb = Kt + (j >> 5) * (C * 32);
#pragma unroll
        for (int k = 0; k < C; k += 16) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int kk = k + half * 8;
            uint32_t x0, x1, x2, x3;
            ldsm4(&s.UsT[arow * SUT + kk + acol], x0, x1, x2, x3);
            mma_tf32(half ? acc2 : acc, x0, x1, x2, x3, raw(kb[swz32(kk + tq, j & 31)]),
                     raw(kb[swz32(kk + tq + 4, j & 31)]));
          }
        }
      }
      if (tid == 0) bulk_wait_read0();   // the chunk-start record has left Sr
      __syncthreads();   // every warp has read S, Sr and Us
      if (upd) {
        const float e0 = acc[0] + acc2[0], e1 = acc[1] + acc2[1];
        const float e2 = acc[2] + acc2[2], e3 = acc[3] + acc2[3];
        s.S[gq * SS + c] = e0;
        s.S[gq * SS + c + 1] = e1;
        s.S[(gq + 8) * SS + c] = e2;
        s.S[(gq + 8) * SS + c + 1] = e3;
        float* sb = s.Sr + (c >> 5) * (BV * 32);
        *reinterpret_cast<float2*>(&sb[swz32(gq, c & 31)]) = make_float2(rnd(e0), rnd(e1));
        *reinterpret_cast<float2*>(&sb[swz32(gq + 8, c & 31)]) = make_float2(rnd(e2), rnd(e3));
      }
      fence_async_smem();   // the next record reads Sr by bulk store
    }
    __syncthreads();
  }
  if (tid == 0) bulk_wait_all0();   // this CTA's records have been written
  if (!ok) {
    // a tile never arrived: wait (bounded) for this CTA's copies in flight, then leave
    if (tid == 0)
      for (int i = 0; i < NS; ++i) {
        bar_wait(&s.full[i], 0);
        bar_wait(&s.full[i], 1);
      }
    __syncthreads();
    return;
  }
  if (sd.ctx_out >= 0) {
    float* So = ctxs[sd.ctx_out].S + head_off;
    for (int i = tid; i < BV * D; i += NTH) {
      const int r = i / D, c = i % D;
      So[(size_t)(v0 + r) * D + c] = s.S[r * SS + c];
    }
  }
}

// ---------------------------------------------------------------------------------------
// chunk_out: one CTA per (chunk, head), 256 threads (8 warps).
// O = diag(gamma) Q S_c^T + P U, P = lower_incl(Gamma * Q K^T); out f16 [R, H*Dv].
// chunk_out: one CTA per (chunk, head, value slice), 256 threads. A CTA forms the output
// columns [vs * D/VS, (vs + 1) * D/VS) of its head; the launcher splits the value columns over
// VS CTAs when (chunks x heads) alone leaves SMs idle (a few questions over a snapshot). P, q's
// norm and (for folded chunks) the whole of W are formed or loaded by every slice.
template <int D, int VS>
struct OutSmem {
  static constexpr int DW = D / VS;  // value columns of the slice
  static constexpr int SQ = D + 4;   // Q, K tiles ([t][j], A / B(n-major) pattern)
  static constexpr int SSC = D + 4;  // chunk-start state rows of the slice ([i][j])
  static constexpr int SUo = D + 8;  // W tile / U slice ([s][i], B k-major pattern)
  static constexpr int SP = C + 4;   // P ([t][s])
  float Q[C * SQ];
  float KU[C * SUo];        // K, then (folded) W, then U
  float S[DW * SSC];
  float P[C * SP];
  float g[C];
};

template <int D, int VS>
__global__ void __launch_bounds__(256) chunk_out_kernel(const float* __restrict__ proj, int ld,
                                                        const float* __restrict__ gbuf,
                                                        const ChunkDesc* __restrict__ chunks, int H, float eps,
                                                        const float* __restrict__ Wbuf,
                                                        const float* __restrict__ Ubuf,
                                                        const float* __restrict__ Schunk,
                                                        const SeqDesc* __restrict__ seqs,
                                                        const CtxDesc* __restrict__ ctxs, int layer_g, int out_fold,
                                                        f16* __restrict__ out) {
  allow_dependents();
  wait_prerequisites();
  extern __shared__ __align__(16) uint8_t smraw[];
  using SM = OutSmem<D, VS>;
  constexpr int SQ = SM::SQ, SSC = SM::SSC, SUo = SM::SUo, SP = SM::SP, DW = SM::DW;
  constexpr int NTO = DW / 16;           // 8-column n-tiles per warp of the output
  SM& s = *reinterpret_cast<SM*>(smraw);
  const int ci = blockIdx.x, h = blockIdx.y, cs = blockIdx.z * DW;
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
  // the slice's rows of the chunk-start state. A folded chunk (a single-chunk sequence without
  // a state pass) starts from the snapshot's state (or zero), TF32-rounded below as the state
  // pass records it.
  const bool fold = cd.seq >= out_fold;
  {
    const float* S0;
    if (!fold) {
      S0 = Schunk + ((size_t)ci * H + h) * D * D;
    } else {
      const int cin = seqs[cd.seq].ctx_in;
      S0 = cin >= 0 ? ctxs[cin].S + (size_t)(layer_g * H + h) * D * D : nullptr;
    }
    for (int i = tid; i < DW * (D / 4); i += 256) {
      const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
      cp16(&s.S[r * SSC + c4], S0 ? S0 + (size_t)(cs + r) * D + c4 : proj, S0 != nullptr);
    }
  }
  if (tid < C) s.g[tid] = tid < n ? gbuf[(size_t)(cd.row0 + tid) * H + h] : 0.f;
  cp_commit();
  cp_wait<0>();
  __syncthreads();
  if (fold) {
    for (int i = tid; i < DW * (D / 4); i += 256) {
      float4* p = reinterpret_cast<float4*>(&s.S[(i / (D / 4)) * SSC + (i % (D / 4)) * 4]);
      const float4 v = *p;
      *p = make_float4(rnd(v.x), rnd(v.y), rnd(v.z), rnd(v.w));
    }
  }
  // q <- q / sqrt(sum q^2 + eps), rounded to TF32 (as k is in chunk_prep); four threads per row
  {
    constexpr int PER = D / 4;
    const int r = tid >> 2, sub = tid & 3;
    float* xs = &s.Q[r * SQ + sub * PER];
    float v[PER];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
      const float4 t = *reinterpret_cast<const float4*>(xs + i);
      v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) ss += v[i] * v[i];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = 1.0f / sqrtf(ss + eps);
#pragma unroll
    for (int i = 0; i < PER; i += 4)
      *reinterpret_cast<float4*>(xs + i) =
          make_float4(rnd(v[i] * inv), rnd(v[i + 1] * inv), rnd(v[i + 2] * inv), rnd(v[i + 3] * inv));
  }
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
  // warp -> rows r0.., value columns cb .. cb + DW/2 of the slice (NTO n-tiles)
  const int cb = (warp >> 2) * (DW / 2);
  if (fold) {
    // U = Ut - W S^T here, with the state pass's TF32 operands (two accumulation chains per
    // output), then rounded to TF32. W (all D key columns) -> KU; Ut straight into registers.
    for (int i = tid; i < C * (D / 4); i += 256) {
      const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
      const bool ok = r < n;
      const int row = cd.row0 + (ok ? r : 0);
      cp16(&s.KU[r * SUo + c4], Wbuf + ((size_t)row * H + h) * D + c4, ok);
    }
    cp_commit();
    float ut[NTO][4];
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      const int c = cs + cb + nt * 8 + 2 * tq;
      const int ra = r0 + gq, rb = r0 + gq + 8;
      const float2 x = ra < n ? *reinterpret_cast<const float2*>(Ubuf + ((size_t)(cd.row0 + ra) * H + h) * D + c)
                              : make_float2(0.f, 0.f);
      const float2 y = rb < n ? *reinterpret_cast<const float2*>(Ubuf + ((size_t)(cd.row0 + rb) * H + h) * D + c)
                              : make_float2(0.f, 0.f);
      ut[nt][0] = x.x; ut[nt][1] = x.y; ut[nt][2] = y.x; ut[nt][3] = y.y;
    }
    cp_wait<0>();
    __syncthreads();
    float u0[NTO][4] = {}, u1[NTO][4] = {};
#pragma unroll 2
    for (int k = 0; k < D; k += 16) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int kk = k + 8 * half;
        const uint32_t a0 = raw(s.KU[(r0 + gq) * SUo + kk + tq]), a1 = raw(s.KU[(r0 + gq + 8) * SUo + kk + tq]);
        const uint32_t a2 = raw(s.KU[(r0 + gq) * SUo + kk + tq + 4]), a3 = raw(s.KU[(r0 + gq + 8) * SUo + kk + tq + 4]);
#pragma unroll
        for (int nt = 0; nt < NTO; ++nt) {
          const int i = cb + nt * 8 + gq;
          const uint32_t b0 = raw(s.S[i * SSC + kk + tq]), b1 = raw(s.S[i * SSC + kk + tq + 4]);
          mma_tf32(half ? u1[nt] : u0[nt], a0, a1, a2, a3, b0, b1);
        }
      }
    }
    __syncthreads();   // every warp has read W
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      const int c = cb + nt * 8 + 2 * tq;
      const int ra = r0 + gq, rb = r0 + gq + 8;
      s.KU[ra * SUo + c] = ra < n ? rnd(ut[nt][0] - (u0[nt][0] + u1[nt][0])) : 0.f;
      s.KU[ra * SUo + c + 1] = ra < n ? rnd(ut[nt][1] - (u0[nt][1] + u1[nt][1])) : 0.f;
      s.KU[rb * SUo + c] = rb < n ? rnd(ut[nt][2] - (u0[nt][2] + u1[nt][2])) : 0.f;
      s.KU[rb * SUo + c + 1] = rb < n ? rnd(ut[nt][3] - (u0[nt][3] + u1[nt][3])) : 0.f;
    }
  } else {
    // the slice of the U tile written by the state pass (k-major stride)
    for (int i = tid; i < C * (DW / 4); i += 256) {
      const int r = i / (DW / 4), c4 = (i % (DW / 4)) * 4;
      const bool ok = r < n;
      const int row = cd.row0 + (ok ? r : 0);
      cp16(&s.KU[r * SUo + c4], Ubuf + ((size_t)row * H + h) * D + cs + c4, ok);
    }
  }
  cp_commit();
  // O1 = Q S_c^T over the slice's value columns
  float o[NTO][4] = {};
#pragma unroll 2
  for (int k = 0; k < D; k += 8) {
    const uint32_t a0 = raw(s.Q[(r0 + gq) * SQ + k + tq]), a1 = raw(s.Q[(r0 + gq + 8) * SQ + k + tq]);
    const uint32_t a2 = raw(s.Q[(r0 + gq) * SQ + k + tq + 4]), a3 = raw(s.Q[(r0 + gq + 8) * SQ + k + tq + 4]);
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      const int i = cb + nt * 8 + gq;
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
      const int i = cb + nt * 8 + gq;
      const uint32_t b0 = raw(s.KU[(k + tq) * SUo + i]), b1 = raw(s.KU[(k + tq + 4) * SUo + i]);
      mma_tf32(o[nt], a0, a1, a2, a3, b0, b1);
    }
  }
  const int HDv = H * D;
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) {
    const int c = cs + cb + nt * 8 + 2 * tq;
    const int ta = r0 + gq, tb = r0 + gq + 8;
    if (ta < n)
      *reinterpret_cast<__half2*>(out + (size_t)(cd.row0 + ta) * HDv + h * D + c) =
          __floats2half2_rn(o[nt][0], o[nt][1]);
    if (tb < n)
      *reinterpret_cast<__half2*>(out + (size_t)(cd.row0 + tb) * HDv + h * D + c) =
          __floats2half2_rn(o[nt][2], o[nt][3]);
  }
}

}  // namespace gc

bool gdn_chunked_supported(int H, int Dk, int Dv, int ld) {
  return Dk == Dv && (Dk == 64 || Dk == 128) && H > 0 && (ld % 4) == 0;
}

template <int D, int NS>
static constexpr size_t state_smem() { return sizeof(gc::StateSmem<D, NS>) + 1024; }

template <int D>
static cudaError_t launch_state(const CUtensorMap& mW, const CUtensorMap& mK, const CUtensorMap& mU,
                                const CUtensorMap& mS, const float* g, const SeqDesc* d_seq, int n_seq, const ChunkDesc* d_chunks,
                                const CtxDesc* d_ctx, int layer_g, int H, float* Ubuf, float* Schunk,
                                int max_chunks, int* d_err, cudaStream_t st) {
  if (n_seq <= 0) return cudaSuccess;
  const dim3 grid(n_seq, H, D / gc::BV);
  if (max_chunks <= 1) {
    CK_RET(launch_pdl(gc::chunk_state_kernel<D, 1>, grid, dim3(512), state_smem<D, 1>(), st, mW, mK, mU, mS, g, d_seq,
                      d_chunks, d_ctx, layer_g, H, Ubuf, Schunk, d_err));
  } else {
    CK_RET(launch_pdl(gc::chunk_state_kernel<D, 2>, grid, dim3(512), state_smem<D, 2>(), st, mW, mK, mU, mS, g, d_seq,
                      d_chunks, d_ctx, layer_g, H, Ubuf, Schunk, d_err));
  }
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_chunked_d(float* proj, int ld, int R, float* loga, float eps, f16* out,
                                    const SeqDesc* d_seq, int n_seq, const ChunkDesc* d_chunks, int n_chunks,
                                    const CtxDesc* d_ctx, int layer_g, int H, float* Wbuf, float* Ubuf,
                                    float* Schunk, int n_first, int max_chunks_first, int max_chunks_rest,
                                    int fold_from, int out_fold, int* d_err, int num_sms, cudaStream_t st) {
  static bool attr = false;
  const size_t sp = sizeof(gc::PrepSmem<D>);
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gc::chunk_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_state_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)state_smem<D, 1>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_state_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)state_smem<D, 2>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_out_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(gc::OutSmem<D, 1>));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_out_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(gc::OutSmem<D, 2>));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_out_kernel<D, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(gc::OutSmem<D, 4>));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CK_RET(launch_pdl(gc::chunk_prep_kernel<D>, dim3(n_chunks, H), dim3(256), sp, st, proj, ld, loga, d_chunks, H, D, eps,
                    Wbuf, Ubuf));
  // TMA views of the chunk tiles: W and Ut rows of head h ([R, H, D] fp32), K columns of proj
  CUtensorMap mW, mK, mU, mS;
  {
    const uint64_t dims3[3] = {(uint64_t)D, (uint64_t)H, (uint64_t)R};
    const uint64_t str3[2] = {(uint64_t)D * 4, (uint64_t)H * D * 4};
    const uint32_t boxW[3] = {32, 1, (uint32_t)gc::C}, boxU[3] = {(uint32_t)gc::BV, 1, (uint32_t)gc::C};
    const uint64_t dims2[2] = {(uint64_t)ld, (uint64_t)R};
    const uint64_t str2[1] = {(uint64_t)ld * 4};
    const uint32_t boxK[2] = {32, (uint32_t)gc::C};
    if (!tensor_map(&mW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, Wbuf, dims3, str3, boxW, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tensor_map(&mU, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, Ubuf, dims3, str3, boxU, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tensor_map(&mK, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, proj, dims2, str2, boxK, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const uint64_t dimsS[2] = {(uint64_t)D, (uint64_t)n_chunks * H * D};
    const uint64_t strS[1] = {(uint64_t)D * 4};
    const uint32_t boxS[2] = {32, (uint32_t)gc::BV};
    if (!tensor_map(&mS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, Schunk, dimsS, strS, boxS, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // sequences [0, n_first) run before the rest (the rest continue from their states). Sequences
  // from fold_from on are followers handled by their prefixes' state pass; sequences from
  // out_fold on are single chunks whose U chunk_out forms itself: neither gets a state pass.
  const int split = (n_first > 0 && n_first < n_seq) ? n_first : n_seq;
  const int n1 = std::min(split, std::min(fold_from, out_fold));
  cudaError_t e = launch_state<D>(mW, mK, mU, mS, loga, d_seq, n1, d_chunks, d_ctx, layer_g, H, Ubuf, Schunk,
                                  split < n_seq ? max_chunks_first : std::max(max_chunks_first, max_chunks_rest),
                                  d_err, st);
  if (e != cudaSuccess) return e;
  const int n2 = std::min(n_seq, out_fold) - split;
  if (split < n_seq && fold_from > split && n2 > 0) {
    e = launch_state<D>(mW, mK, mU, mS, loga, d_seq + split, n2, d_chunks, d_ctx, layer_g, H, Ubuf, Schunk,
                        max_chunks_rest, d_err, st);
    if (e != cudaSuccess) return e;
  }
  // value columns split over 2 or 4 CTAs while (chunks x heads) CTAs leave SMs idle
  int vs = 1;
  while (vs < 4 && (long)n_chunks * H * vs < num_sms) vs *= 2;
  switch (vs) {
    case 1:
      CK_RET(launch_pdl(gc::chunk_out_kernel<D, 1>, dim3(n_chunks, H, 1), dim3(256), sizeof(gc::OutSmem<D, 1>), st,
                        proj, ld, loga, d_chunks, H, eps, Wbuf, Ubuf, Schunk, d_seq, d_ctx, layer_g, out_fold, out));
      break;
    case 2:
      CK_RET(launch_pdl(gc::chunk_out_kernel<D, 2>, dim3(n_chunks, H, 2), dim3(256), sizeof(gc::OutSmem<D, 2>), st,
                        proj, ld, loga, d_chunks, H, eps, Wbuf, Ubuf, Schunk, d_seq, d_ctx, layer_g, out_fold, out));
      break;
    default:
      CK_RET(launch_pdl(gc::chunk_out_kernel<D, 4>, dim3(n_chunks, H, 4), dim3(256), sizeof(gc::OutSmem<D, 4>), st,
                        proj, ld, loga, d_chunks, H, eps, Wbuf, Ubuf, Schunk, d_seq, d_ctx, layer_g, out_fold, out));
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_gdn_chunked(float* proj, int ld, int R, float* loga, float eps, f16* out,
                               const SeqDesc* d_seq, int n_seq, const ChunkDesc* d_chunks, int n_chunks,
                               const CtxDesc* d_ctx, int layer_g, int H, int Dk, int Dv, float* Wbuf, float* Ubuf,
                               float* Schunk, int n_first, int max_chunks_first, int max_chunks_rest,
                               int fold_from, int out_fold, int* d_err, int num_sms, cudaStream_t st,
                               long* launches) {
  if (n_seq <= 0 || n_chunks <= 0) return cudaSuccess;
  if (!gdn_chunked_supported(H, Dk, Dv, ld)) return cudaErrorNotSupported;
  if (n_seq > 65535 || n_chunks > 2147483647 / 2) return cudaErrorInvalidValue;
  cudaError_t e = (Dk == 128)
                      ? launch_chunked_d<128>(proj, ld, R, loga, eps, out, d_seq, n_seq, d_chunks, n_chunks, d_ctx,
                                              layer_g, H, Wbuf, Ubuf, Schunk, n_first, max_chunks_first,
                                              max_chunks_rest, fold_from, out_fold, d_err, num_sms, st)
                      : launch_chunked_d<64>(proj, ld, R, loga, eps, out, d_seq, n_seq, d_chunks, n_chunks, d_ctx,
                                             layer_g, H, Wbuf, Ubuf, Schunk, n_first, max_chunks_first,
                                             max_chunks_rest, fold_from, out_fold, d_err, num_sms, st);
  if (launches) {
    const int split = (n_first > 0 && n_first < n_seq) ? n_first : n_seq;
    *launches += 2 + (std::min(split, std::min(fold_from, out_fold)) > 0 ? 1 : 0) +
                 (split < n_seq && fold_from > split && std::min(n_seq, out_fold) > split ? 1 : 0);
  }
  return e;
}

}  // namespace s1
