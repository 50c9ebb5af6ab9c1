// Chunked gated delta rule (WY form) for prefill-length sequences.
//
// For a chunk of n <= 64 rows with state S0 at its start ([Dv, Dk] per head), with
// g = cumsum(log alpha) inside the chunk, gamma = exp(g), Gamma_ts = exp(g_t - g_s):
//   A  = strict_lower(diag(beta) (Gamma * K K^T)),   T = (I + A)^-1
//   W  = T diag(beta gamma) K,    Ut = T diag(beta) V
//   U  = Ut - W S0^T                                  (the delta-rule write vectors)
//   O  = diag(gamma) Q S0^T + lower_incl(Gamma * Q K^T) U
//   S_next = gamma_n S0 + U^T K',   K'_t = exp(g_n - g_t) k_t
// (WY representation of the gated delta rule, Yang, Kautz & Hatamizadeh, "Gated Delta
// Networks", 2024; it reaches the token recurrence's result up to rounding, which the pages
// allow for chunk boundaries: System1-Omni RFC #114, section 5.)
//
// With U substituted, a chunk's state step is affine in its start state:
//   S_next = gamma_n S0 - S0 N + B,    N = W^T K' [Dk, Dk],   B = Ut^T K' [Dv, Dk]
// N depends on the chunk's own rows only, so chunk_prep forms it in parallel with the rest of
// the chunk's algebra; B is formed by the state pass off its critical path. What has to run
// chunk after chunk is one [16, Dk] x [Dk, Dk] product per 16 state rows and chunk (the state
// itself stays fp32, in registers).
//
// Launches per layer (the gates and the q/k L2 norms are formed inside them):
//   chunk_prep  (chunk, head)             gates, k norm, g, A, forward substitution for W and
//                                         Ut, then K' and N^T                      (parallel)
//   chunk_state (sequence, head, 16 rows) S <- gamma_n S + Ut^T K' - S N per chunk; records
//                                         every chunk's start state             (sequential)
//   chunk_out   (chunk, head, v slice)    q norm, P, U = Ut - W S_c^T, O = gamma Q S_c^T + P U
//                                                                                 (parallel)
// Single-chunk sequences that keep no state need no state step: in a one-sweep call the
// prefix's state pass records their start state (its own final state); otherwise chunk_out
// reads their start state from the snapshot. Every product runs on the tensor cores as
// mma.sync m16n8k16 with f16 operands (the 10-bit mantissa of TF32) and fp32 accumulation.
#include <algorithm>

#include "common.cuh"

namespace s1 {
namespace gc {

constexpr int C = 64;      // chunk rows
constexpr int BV = 16;     // state rows per state-pass CTA
constexpr int NS = 4;      // chunk tiles in flight per state-pass CTA
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

// D += A(16x16, row) * B(16x8, col): f16 inputs, fp32 accumulate
__device__ __forceinline__ void mma16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t h2u(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Fragment loads from f16 tiles in shared memory with a row stride of `ld` halves (ld * 2 bytes
// = 16 mod 128 keeps the eight rows of each ldmatrix phase on distinct banks).
// A operand (16 x 16) at (m0, k0) of a tile stored [m][k].
__device__ __forceinline__ void lda(const __half* t, int ld, int m0, int k0, int lane, uint32_t* a) {
  ldsm4(smem_u32(t + (m0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * ld + k0 + 8 * (lane >> 4)), a);
}
// A operand (16 x 16) at (m0, k0) of a tile stored transposed, [k][m].
__device__ __forceinline__ void lda_t(const __half* t, int ld, int m0, int k0, int lane, uint32_t* a) {
  ldsm4t(smem_u32(t + (k0 + (lane & 7) + 8 * (lane >> 4)) * ld + m0 + 8 * ((lane >> 3) & 1)), a);
}
// B operands of the n-tile at n0 over k0 .. k0+31 of a tile stored [n][k]: {b0, b1} of
// k0 .. k0+15, then of k0+16 .. k0+31.
__device__ __forceinline__ void ldb_nk(const __half* t, int ld, int n0, int k0, int lane, uint32_t* b) {
  ldsm4(smem_u32(t + (n0 + (lane & 7)) * ld + k0 + 8 * (lane >> 3)), b);
}
// B operands of the n-tiles at n0 and n0+8 over k0 .. k0+15 of a tile stored [k][n]:
// {b0, b1} of the first n-tile, then of the second.
__device__ __forceinline__ void ldb_kn2(const __half* t, int ld, int n0, int k0, int lane, uint32_t* b) {
  ldsm4t(smem_u32(t + (k0 + (lane & 15)) * ld + n0 + 8 * (lane >> 4)), b);
}

// Rows r < n of a chunk load 4 floats per call (zeros past n).
__device__ __forceinline__ float4 ld4(const float* src, bool ok) {
  return ok ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------------------
// chunk_prep: one CTA per (chunk, head), 256 threads (8 warps), two CTAs per SM.
// Writes g (within-chunk cumsum of log alpha), the normalised k, W and Ut (f16 [R, H, D]) and,
// when a state pass takes a step over this chunk, K' (f16 [R, H, D]), N^T (f16 [chunks, H, D, D])
// and gamma_n.
// The unit-lower-triangular system (I + A) X = [diag(beta gamma) K | diag(beta) V] is solved in
// 16-row blocks: each 16 x 16 diagonal block's inverse T_bb comes from forward substitution in
// fp32 (one thread per column), then X_b = T_bb (RHS_b - sum_{c<b} A_bc X_c) on the tensor cores.
template <int D>
struct PrepSmem {
  static constexpr int SK = D + 8;         // f16 stride of D-wide tiles
  static constexpr int SX = 2 * D + 8;     // f16 stride of X = [W | Ut]
  static constexpr int SA = C + 4;         // fp32 A
  static constexpr int SAH = C + 8;        // f16 A
  static constexpr int ST = 24;            // f16 diagonal-block inverses
  __half Kh[C * SK];                       // normalised k
  __half X[C * SX];
  __half Ah[C * SAH];
  __half T[4][16 * ST];
  float A[C * SA];
  struct {
    __half Kp[C * SK];                     // K'_t = exp(g_n - g_t) k_t (after the solve)
  } u;
  float g[C];
  float b[C];
  float la[C];                             // log alpha
};

// SPLIT: the chunks need no state step (questions that continue a snapshot) and the right-hand
// side is split over two CTAs per (chunk, head): blockIdx.z = 0 solves for W (and writes the
// normalised k and g), 1 for Ut; both form A and its diagonal-block inverses.
template <int D, bool SPLIT = false>
__global__ void __launch_bounds__(256, 2) chunk_prep_kernel(const float* __restrict__ proj, int ld,
                                                            float* __restrict__ gout,
                                                            const ChunkDesc* __restrict__ chunks,
                                                            const SeqDesc* __restrict__ seqs, int H, float eps,
                                                            GdnBufs bufs) {
  allow_dependents();
  wait_prerequisites();
  using SM = PrepSmem<D>;
  const int half = SPLIT ? (int)blockIdx.z : 0;
  constexpr int SK = SM::SK, SX = SM::SX, SA = SM::SA, SAH = SM::SAH, ST = SM::ST;
  constexpr int PER = D / 4;               // columns per thread in the row-wise phases
  extern __shared__ __align__(16) uint8_t smraw[];
  SM& s = *reinterpret_cast<SM*>(smraw);
  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const ChunkDesc cd = chunks[ci];
  const int n = cd.len;
  const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int HD = H * D;
  // a state pass steps over this chunk unless it is the last chunk of a sequence whose final
  // state nobody keeps
  bool need_nb;
  {
    const SeqDesc sd = seqs[cd.seq];
    need_nb = cd.row0 + n != sd.row0 + sd.len || sd.ctx_out >= 0 || sd.fol1 > sd.fol0;
  }
  // this thread's quarter of row r of k and v (rows past n read as zero)
  const int r = tid >> 2, c0 = (tid & 3) * PER;
  float kv[PER], vv[PER];
  {
    const bool ok = r < n;
    const float* pr = proj + (size_t)(cd.row0 + (ok ? r : 0)) * ld + h * D + c0;
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
      const float4 a = ld4(pr + HD + i, ok), b = ld4(pr + 2 * HD + i, ok);
      kv[i] = a.x; kv[i + 1] = a.y; kv[i + 2] = a.z; kv[i + 3] = a.w;
      vv[i] = b.x; vv[i + 1] = b.y; vv[i + 2] = b.z; vv[i + 3] = b.w;
    }
  }
  if (tid < C) {
    // alpha_t = exp(-softplus(a_t)), beta_t = sigmoid(b_t)
    float la = 0.f, bt = 0.f;
    if (tid < n) {
      const float* ab = proj + (size_t)(cd.row0 + tid) * ld + 3 * HD;
      const float a = ab[h], b = ab[H + h];
      la = -(fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))));
      bt = 1.f / (1.f + expf(-b));
    }
    s.la[tid] = la;
    s.b[tid] = bt;
  }
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
  __syncthreads();
  // k <- k / sqrt(sum k^2 + eps); right-hand sides beta gamma k | beta v (four threads per row)
  {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) ss += kv[i] * kv[i];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = 1.0f / sqrtf(ss + eps);
    const float bt = s.b[r], wsc = bt * __expf(s.g[r]);
    f16* kg = bufs.Kn + ((size_t)(cd.row0 + r) * H + h) * D + c0;
#pragma unroll
    for (int i = 0; i < PER; i += 8) {
      uint32_t kk[4], ww[4], uu[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float k0 = kv[i + 2 * j] * inv, k1 = kv[i + 2 * j + 1] * inv;
        kk[j] = h2u(k0, k1);
        ww[j] = h2u(k0 * wsc, k1 * wsc);
        uu[j] = h2u(vv[i + 2 * j] * bt, vv[i + 2 * j + 1] * bt);
      }
      *reinterpret_cast<uint4*>(&s.Kh[r * SK + c0 + i]) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
      if constexpr (SPLIT) {   // this CTA's half of the right-hand side, in X's first D columns
        *reinterpret_cast<uint4*>(&s.X[r * SX + c0 + i]) =
            half ? make_uint4(uu[0], uu[1], uu[2], uu[3]) : make_uint4(ww[0], ww[1], ww[2], ww[3]);
      } else {
        *reinterpret_cast<uint4*>(&s.X[r * SX + c0 + i]) = make_uint4(ww[0], ww[1], ww[2], ww[3]);
        *reinterpret_cast<uint4*>(&s.X[r * SX + D + c0 + i]) = make_uint4(uu[0], uu[1], uu[2], uu[3]);
      }
      if (r < n && half == 0) *reinterpret_cast<uint4*>(kg + i) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
    }
  }
  __syncthreads();
  // ---- A = strict_lower(beta_t exp(g_t - g_s) k_t.k_s): warp -> m-tile (warp & 3), 4 n-tiles.
  // Only the strictly lower part is ever read (the diagonal blocks' inverses and the blocks left
  // of them), so the two warps whose tiles lie wholly above the diagonal skip theirs.
  if ((warp >> 2) * 32 <= (warp & 3) * 16 + 15) {
    const int m0 = (warp & 3) * 16, nb = (warp >> 2) * 32;
    float acc[4][4] = {};
#pragma unroll
    for (int k = 0; k < D; k += 32) {
      uint32_t a0[4], a1[4];
      lda(s.Kh, SK, m0, k, lane, a0);
      lda(s.Kh, SK, m0, k + 16, lane, a1);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t b[4];
        ldb_nk(s.Kh, SK, nb + nt * 8, k, lane, b);
        mma16(acc[nt], a0, b[0], b[1]);
        mma16(acc[nt], a1, b[2], b[3]);
      }
    }
    const int ta = m0 + gq, tb = ta + 8;       // this thread's rows; columns c, c + 1 per n-tile
    const float ga = s.g[ta], gb = s.g[tb], ba = s.b[ta], bb = s.b[tb];
    const bool oka = ta < n, okb = tb < n;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = nb + nt * 8 + 2 * tq;
      const float g0 = s.g[c], g1 = s.g[c + 1];
      const float va0 = (oka && c < ta) ? ba * __expf(ga - g0) * acc[nt][0] : 0.f;
      const float va1 = (oka && c + 1 < ta) ? ba * __expf(ga - g1) * acc[nt][1] : 0.f;
      const float vb0 = (okb && c < tb) ? bb * __expf(gb - g0) * acc[nt][2] : 0.f;
      const float vb1 = (okb && c + 1 < tb) ? bb * __expf(gb - g1) * acc[nt][3] : 0.f;
      *reinterpret_cast<float2*>(&s.A[ta * SA + c]) = make_float2(va0, va1);
      *reinterpret_cast<float2*>(&s.A[tb * SA + c]) = make_float2(vb0, vb1);
      *reinterpret_cast<uint32_t*>(&s.Ah[ta * SAH + c]) = h2u(va0, va1);
      *reinterpret_cast<uint32_t*>(&s.Ah[tb * SAH + c]) = h2u(vb0, vb1);
    }
  }
  __syncthreads();
  // ---- diagonal-block inverses T_bb = (I + N_bb)^-1, N_bb the strictly lower 16 x 16 diagonal
  // block of A: forward substitution in fp32, one thread per (block, column j):
  // x_i = [i == j] - sum_{k < i} N_ik x_k (rows i < j come out zero)
  if (tid < 64) {
    const int bb = tid >> 4, j = tid & 15;
    const float* Nb = s.A + bb * 16 * SA + bb * 16;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a0 = i == j ? 1.f : 0.f, a1 = 0.f;   // two partial sums: shorter dependent chains
#pragma unroll
      for (int k = 0; k + 1 < i; k += 2) {
        a0 = fmaf(-Nb[i * SA + k], x[k], a0);
        a1 = fmaf(-Nb[i * SA + k + 1], x[k + 1], a1);
      }
      if (i & 1) a0 = fmaf(-Nb[i * SA + i - 1], x[i - 1], a0);
      x[i] = a0 + a1;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) s.T[bb][i * ST + j] = __float2half_rn(x[i]);
  }
  __syncthreads();
  // ---- block forward substitution over the 4 row blocks; each warp owns NT n-tiles of X
  constexpr int NT = (SPLIT ? 1 : 2) * D / 64;   // n-tiles per warp (D = 128: 4, D = 64: 2; halved when split)
  const int cw = warp * NT * 8;            // this warp's first column of X
  for (int bb = 0; bb < 4; ++bb) {
    const int r0 = bb * 16;
    float acc[NT][4], sub[NT][4] = {};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = cw + nt * 8 + 2 * tq;
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&s.X[(r0 + gq) * SX + c]));
      const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&s.X[(r0 + gq + 8) * SX + c]));
      acc[nt][0] = x.x; acc[nt][1] = x.y; acc[nt][2] = y.x; acc[nt][3] = y.y;
    }
    // R_b = RHS_b - A[b, 0:16b] X[0:16b]
    for (int k = 0; k < r0; k += 16) {
      uint32_t a[4];
      lda(s.Ah, SAH, r0, k, lane, a);
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        uint32_t b[4];
        ldb_kn2(s.X, SX, cw + nt * 8, k, lane, b);
        mma16(sub[nt], a, b[0], b[1]);
        mma16(sub[nt + 1], a, b[2], b[3]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = cw + nt * 8 + 2 * tq;
      *reinterpret_cast<uint32_t*>(&s.X[(r0 + gq) * SX + c]) = h2u(acc[nt][0] - sub[nt][0], acc[nt][1] - sub[nt][1]);
      *reinterpret_cast<uint32_t*>(&s.X[(r0 + gq + 8) * SX + c]) =
          h2u(acc[nt][2] - sub[nt][2], acc[nt][3] - sub[nt][3]);
    }
    __syncwarp();
    // X_b = T_bb R_b
    float xb[NT][4] = {};
    {
      uint32_t a[4];
      lda(s.T[bb], ST, 0, 0, lane, a);
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        uint32_t b[4];
        ldb_kn2(s.X, SX, cw + nt * 8, r0, lane, b);
        mma16(xb[nt], a, b[0], b[1]);
        mma16(xb[nt + 1], a, b[2], b[3]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int c = cw + nt * 8 + 2 * tq;
      *reinterpret_cast<uint32_t*>(&s.X[(r0 + gq) * SX + c]) = h2u(xb[nt][0], xb[nt][1]);
      *reinterpret_cast<uint32_t*>(&s.X[(r0 + gq + 8) * SX + c]) = h2u(xb[nt][2], xb[nt][3]);
    }
    __syncwarp();
  }
  __syncthreads();
  // W and Ut rows (16-byte pieces) and g
  if constexpr (SPLIT) {
    for (int i = tid; i < n * (D / 8); i += 256) {
      const int rr = i / (D / 8), c8 = (i % (D / 8)) * 8;
      const uint4 v = *reinterpret_cast<const uint4*>(&s.X[rr * SX + c8]);
      const size_t o = ((size_t)(cd.row0 + rr) * H + h) * D;
      *reinterpret_cast<uint4*>((half ? bufs.Ut : bufs.W) + o + c8) = v;
    }
    if (tid < n && half == 0) gout[(size_t)(cd.row0 + tid) * H + h] = s.g[tid];
  } else {
    for (int i = tid; i < n * (2 * D / 8); i += 256) {
      const int rr = i / (2 * D / 8), c8 = (i % (2 * D / 8)) * 8;
      const uint4 v = *reinterpret_cast<const uint4*>(&s.X[rr * SX + c8]);
      const size_t o = ((size_t)(cd.row0 + rr) * H + h) * D;
      *reinterpret_cast<uint4*>(c8 < D ? bufs.W + o + c8 : bufs.Ut + o + c8 - D) = v;
    }
    if (tid < n) gout[(size_t)(cd.row0 + tid) * H + h] = s.g[tid];
  }
  // (split chunks take no state step: no K', N^T or gamma_n)
  if (SPLIT || !need_nb) return;
  // ---- K'_t = exp(g_n - g_t) k_t (into shared memory and to global), gamma_n
  {
    const float gl = s.g[n - 1];
    for (int i = tid; i < C * (D / 8); i += 256) {
      const int rr = i / (D / 8), c = (i % (D / 8)) * 8;
      const float e = rr < n ? __expf(gl - s.g[rr]) : 0.f;
      const uint4 kq = *reinterpret_cast<const uint4*>(&s.Kh[rr * SK + c]);
      const __half2* kh = reinterpret_cast<const __half2*>(&kq);
      uint32_t w[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const float2 k = __half22float2(kh[e2]);
        w[e2] = h2u(k.x * e, k.y * e);
      }
      const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(&s.u.Kp[rr * SK + c]) = v;
      if (rr < n) *reinterpret_cast<uint4*>(bufs.Kp + ((size_t)(cd.row0 + rr) * H + h) * D + c) = v;
    }
    if (tid == 0) bufs.gam[(size_t)ci * H + h] = __expf(gl);
  }
  __syncthreads();
  // ---- N^T = K'^T W ([D, D]); warp -> m-tile, NPW n-tiles; staged in shared memory (over the
  // normalised k and X, no longer read) and written out in 16-byte pieces
  {
    constexpr int MT = D / 16, NG = 8 / MT, NPW = (D / 8) / NG, SN = D + 8;
    static_assert(D * SN * 2 <= (int)(sizeof(s.Kh) + sizeof(s.X)), "N^T staging exceeds the free space");
    const int m0 = (warp % MT) * 16, n0 = (warp / MT) * NPW * 8;
    float acc[NPW][4];
#pragma unroll
    for (int j = 0; j < NPW; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
    for (int k = 0; k < C; k += 16) {
      uint32_t a[4];
      lda_t(s.u.Kp, SK, m0, k, lane, a);
#pragma unroll
      for (int j = 0; j < NPW; j += 2) {
        uint32_t b[4];
        ldb_kn2(s.X, SX, n0 + j * 8, k, lane, b);
        mma16(acc[j], a, b[0], b[1]);
        mma16(acc[j + 1], a, b[2], b[3]);
      }
    }
    __syncthreads();   // every warp has read X and K'
    __half* stg = s.Kh;
#pragma unroll
    for (int j = 0; j < NPW; ++j) {
      const int c = n0 + j * 8 + 2 * tq;
      *reinterpret_cast<uint32_t*>(&stg[(m0 + gq) * SN + c]) = h2u(acc[j][0], acc[j][1]);
      *reinterpret_cast<uint32_t*>(&stg[(m0 + gq + 8) * SN + c]) = h2u(acc[j][2], acc[j][3]);
    }
    __syncthreads();
    f16* dst = bufs.NT + ((size_t)ci * H + h) * D * D;
    for (int i = tid; i < D * (D / 8); i += 256) {
      const int rr = i / (D / 8), c = (i % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(dst + (size_t)rr * D + c) = *reinterpret_cast<const uint4*>(&stg[rr * SN + c]);
    }
  }
}

// ---------------------------------------------------------------------------------------
// chunk_state: one CTA per (sequence, head, block of 16 state rows), D / 16 warps; warp w keeps
// columns [16w, 16w + 16) of the block's fp32 state in registers (two m16n8 accumulators). Per
// chunk: S <- gamma_n S + Ut_b^T K' - Sr N, Sr the f16 copy of S in shared memory (all warps'
// columns, the A operand of the product that depends on the previous chunk), Ut_b the block's
// 16 columns of Ut. Each chunk's N^T, K' and Ut_b tiles arrive by TMA (one thread issues them
// up to NS chunks ahead; every wait is bounded); its start state is recorded (f16) for
// chunk_out.
template <int D, int NST>
struct StateSmem {
  static constexpr int SR = D + 8;
  static constexpr int NT_BYTES = D * D * 2;       // D / 64 boxes of [D rows][64 columns], swizzled
  static constexpr int KP_BYTES = C * D * 2;       // D / 64 boxes of [64 rows][64 columns], swizzled
  static constexpr int UT_BYTES = C * BV * 2;      // [64 rows][16 columns], dense
  static constexpr int STAGE = NT_BYTES + KP_BYTES + UT_BYTES;
  static constexpr int GAM = 256;                  // gamma_n of up to this many chunks at a time
  uint8_t stage[NST][STAGE];
  __half Sr[2][BV * SR];
  float gam[GAM];
  uint64_t full[NST];
};

// element offset of (row, col) in a swizzled N^T tile
template <int D>
__device__ __forceinline__ int nt_off(int row, int col) {
  return (col >> 6) * (D * 64) + row * 64 + ((((col & 63) >> 3) ^ (row & 7)) << 3) + (col & 7);
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

// mapNT: N^T [n_chunks * H * D rows, D columns] f16, box 64 x D, 128-byte swizzle.
// mapKp: K' [R, H, D] f16 as (D, H, R), box 64 x 1 x 64, 128-byte swizzle.
// mapUt: Ut [R, H, D] f16 as (D, H, R), box 16 x 1 x 64, no swizzle.
// Threads of the state pass: one warp per 16 state columns.
template <int D>
constexpr int state_threads() { return D * 2; }

// NST chunk tiles in flight: 4 while the CTAs fit one wave (one CTA per SM), 2 when they need
// several (two CTAs per SM, at most 128 registers a thread).
template <int D, int NST>
__global__ void __launch_bounds__(D * 2, NST == 2 ? 2 : 1) chunk_state_kernel(const __grid_constant__ CUtensorMap mapNT,
                                                            const __grid_constant__ CUtensorMap mapKp,
                                                            const __grid_constant__ CUtensorMap mapUt,
                                                            const float* __restrict__ gam,
                                                            const SeqDesc* __restrict__ seqs,
                                                            const ChunkDesc* __restrict__ chunks,
                                                            const CtxDesc* __restrict__ ctxs, int layer_g, int H,
                                                            f16* __restrict__ Srec, int* __restrict__ d_err) {
  allow_dependents();
  wait_prerequisites();
  using SM = StateSmem<D, NST>;
  constexpr int SR = SM::SR;
  constexpr int KS = D / 32;                   // 32-deep k steps of Sr x N
  extern __shared__ __align__(16) uint8_t smraw[];   // (rounded up to 1024 bytes below)
  SM& s = *reinterpret_cast<SM*>((((uintptr_t)smraw) + 1023) & ~(uintptr_t)1023);
  const SeqDesc sd = seqs[blockIdx.x];
  const int h = blockIdx.y, v0 = blockIdx.z * BV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int nch = (sd.len + C - 1) / C;
  // steps that update the state: all but the last chunk's, unless the final state is kept
  const int nupd = (sd.ctx_out >= 0 || sd.fol1 > sd.fol0) ? nch : nch - 1;
  const int cw = warp * 16;                    // this warp's state columns cw .. cw + 15
  const size_t DD = (size_t)D * D;
  const size_t head_off = (size_t)(layer_g * H + h) * DD;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) bar_init(&s.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  int issued = 0;                              // steps whose tiles were requested (warp 0)
  // warp 0 requests a step's tiles: lane 0 sets the byte count, then one copy per lane (the
  // D / 64 boxes of N^T and of K', and the Ut block)
  auto issue = [&](int cl, int ln) {
    const int st = cl % NST;
    uint8_t* sb = s.stage[st];
    if (ln == 0) bar_expect_tx(&s.full[st], SM::STAGE);
    __syncwarp();
    const int ci = sd.chunk0 + cl;
    const int row0 = sd.row0 + cl * C;         // the chunk's first packed row
    constexpr int NB = D / 64;
    if (ln < NB) tma2(sb + ln * D * 128, &mapNT, &s.full[st], 64 * ln, (ci * H + h) * D);
    else if (ln < 2 * NB) tma3(sb + SM::NT_BYTES + (ln - NB) * C * 128, &mapKp, &s.full[st], 64 * (ln - NB), h, row0);
    else if (ln == 2 * NB) tma3(sb + SM::NT_BYTES + SM::KP_BYTES, &mapUt, &s.full[st], v0, h, row0);
    ++issued;
  };
  if (warp == 0)
    for (int cl = 0; cl < nupd && cl < NST; ++cl) issue(cl, lane);
  // gamma_n of the first steps
  for (int i = tid; i < nupd && i < SM::GAM; i += blockDim.x) s.gam[i] = gam[(size_t)(sd.chunk0 + i) * H + h];
  // the state block's fragments: rows v0 + gq and v0 + gq + 8, columns cw + 8 nt + 2 tq and + 1
  float acc[2][4] = {};
  if (sd.ctx_in >= 0) {
    const float* S0 = ctxs[sd.ctx_in].S + head_off;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = cw + 8 * nt + 2 * tq;
      const float2 x = *reinterpret_cast<const float2*>(S0 + (size_t)(v0 + gq) * D + col);
      const float2 y = *reinterpret_cast<const float2*>(S0 + (size_t)(v0 + gq + 8) * D + col);
      acc[nt][0] = x.x; acc[nt][1] = x.y; acc[nt][2] = y.x; acc[nt][3] = y.y;
    }
  }
  // f16 copy of the fragments into Sr[buf], and into the start record of chunk ci (ci >= 0)
  auto put = [&](int buf, int ci) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = cw + 8 * nt + 2 * tq;
      const uint32_t lo = h2u(acc[nt][0], acc[nt][1]), hi = h2u(acc[nt][2], acc[nt][3]);
      *reinterpret_cast<uint32_t*>(&s.Sr[buf][gq * SR + col]) = lo;
      *reinterpret_cast<uint32_t*>(&s.Sr[buf][(gq + 8) * SR + col]) = hi;
      if (ci >= 0) {
        f16* rp = Srec + ((size_t)ci * H + h) * DD;
        *reinterpret_cast<uint32_t*>(rp + (size_t)(v0 + gq) * D + col) = lo;
        *reinterpret_cast<uint32_t*>(rp + (size_t)(v0 + gq + 8) * D + col) = hi;
      }
    }
  };
  put(0, sd.chunk0);
  // Everything a step needs from its tiles is taken during the step before it, while that step's
  // Sr x N products are in flight: the B block = Ut_b^T K' over this warp's 16 columns
  // (independent of the state; rows t >= n of both tiles are zeroed in the fragments), kept in
  // qv, and this warp's N fragments, kept in nb (qv2 / nb2 for the next step). After the barrier
  // a step is only Sr x N, the update and the f16 copy.
  float qv[2][4], qv2[2][4];
  uint32_t nb[KS][2][4], nb2[KS][2][4];
  auto take_tiles = [&](int cl, float (&qo)[2][4], uint32_t (&no)[KS][2][4]) {
    const uint8_t* sb = s.stage[cl % NST];
    const __half* ntile = reinterpret_cast<const __half*>(sb);
    const uint32_t kp_base = smem_u32(sb + SM::NT_BYTES);
    const __half* ut = reinterpret_cast<const __half*>(sb + SM::NT_BYTES + SM::KP_BYTES);
    const int n = min(C, sd.len - cl * C);     // rows of this chunk (later tile rows belong to others
                                               // or, past the call's rows, hold whatever the scratch held)
    float q[2][2][4] = {};
#pragma unroll
    for (int k = 0; k < C; k += 32) {
      uint32_t a0[4], a1[4];
      lda_t(ut, BV, 0, k, lane, a0);
      lda_t(ut, BV, 0, k + 16, lane, a1);
      if (n < C) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t0 = k + ((e >> 1) << 3) + 2 * tq, t1 = t0 + 16;
          const uint32_t m0 = (t0 < n ? 0x0000FFFFu : 0u) | (t0 + 1 < n ? 0xFFFF0000u : 0u);
          const uint32_t m1 = (t1 < n ? 0x0000FFFFu : 0u) | (t1 + 1 < n ? 0xFFFF0000u : 0u);
          a0[e] &= m0;
          a1[e] &= m1;
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        // K' rows k .. k+31 (token), 8 columns of this warp; swizzled boxes of 64 columns;
        // b[j] holds tokens k + 8j + 2tq and + 1
        uint32_t b[4];
        const int t = k + lane, c = cw + 8 * nt;
        ldsm4t(kp_base + (uint32_t)((c >> 6) * (C * 128) + t * 128 + ((((c & 63) >> 3) ^ (t & 7)) << 4)), b);
        if (n < C) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int t0 = k + 8 * j + 2 * tq;
            b[j] &= (t0 < n ? 0x0000FFFFu : 0u) | (t0 + 1 < n ? 0xFFFF0000u : 0u);
          }
        }
        mma16(q[nt][0], a0, b[0], b[1]);
        mma16(q[nt][1], a1, b[2], b[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) qo[nt][i] = q[nt][0][i] + q[nt][1][i];
#pragma unroll
    for (int i = 0; i < KS; ++i)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        ldsm4(smem_u32(ntile + nt_off<D>(cw + 8 * nt + (lane & 7), 32 * i + 8 * (lane >> 3))), no[i][nt]);
  };
  // the first tiles; one barrier agrees on their arrival and on Sr and gamma being in place
  bool ok = __syncthreads_and(nupd > 0 ? (bar_wait(&s.full[0], 0) ? 1 : 0) : 1) != 0;
  int waited = (ok && nupd > 0) ? 1 : 0;     // steps whose tiles have arrived
  if (ok && nupd > 0) take_tiles(0, qv, nb);
  int cur = 0;
  for (int cl = 0; cl < nupd && ok; ++cl) {
    // Sr (16 x D) x N (D x D) over this warp's 16 columns: the A fragments are shared by both
    // column tiles; two accumulation chains per tile
    float p[2][2][4] = {};
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      uint32_t a0[4], a1[4];
      lda(s.Sr[cur], SR, 0, 32 * i, lane, a0);
      lda(s.Sr[cur], SR, 0, 32 * i + 16, lane, a1);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma16(p[nt][i & 1], a0, nb[i][nt][0], nb[i][nt][1]);
        mma16(p[nt][i & 1], a1, nb[i][nt][2], nb[i][nt][3]);
      }
    }
    // the next step's tiles, taken while those products complete
    bool w = true;
    if (cl + 1 < nupd) {
      w = bar_wait(&s.full[(cl + 1) % NST], ((cl + 1) / NST) & 1);
      if (w) take_tiles(cl + 1, qv2, nb2);
    }
    const float g = s.gam[cl % SM::GAM];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = fmaf(g, acc[nt][i], qv[nt][i] - (p[nt][0][i] + p[nt][1][i]));
    put(cur ^ 1, cl + 1 < nch ? sd.chunk0 + cl + 1 : -1);
    // one barrier that agrees on the next step's tiles, on Sr being complete and on the tiles
    // of this step and the next having been read by every warp
    ok = __syncthreads_and(w ? 1 : 0) != 0;
    if (!ok) break;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[nt][i] = qv2[nt][i];
#pragma unroll
    for (int i = 0; i < KS; ++i)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) nb[i][nt][j] = nb2[i][nt][j];
    if (cl + 1 < nupd) ++waited;
    if (warp == 0 && cl + NST < nupd) issue(cl + NST, lane);   // refill the stage this step consumed
    cur ^= 1;
    if ((cl + 1) % SM::GAM == 0 && cl + 1 < nupd) {   // the next block of gamma_n
      for (int i = tid; i < SM::GAM && cl + 1 + i < nupd; i += blockDim.x)
        s.gam[i] = gam[(size_t)(sd.chunk0 + cl + 1 + i) * H + h];
      __syncthreads();
    }
  }
  if (!ok) {
    // a tile never arrived: wait (bounded) for this CTA's copies in flight, then leave
    if (tid == 0) {
      atomicExch(d_err, 0x201);
      for (int j = waited; j < issued; ++j) bar_wait(&s.full[j % NST], (j / NST) & 1);
    }
    __syncthreads();
    return;
  }
  // the final state: start record of every follower, and the snapshot
  if (nupd == nch) {
    for (int f = sd.fol0; f < sd.fol1; ++f) put(cur, seqs[f].chunk0);
    if (sd.ctx_out >= 0) {
      float* So = ctxs[sd.ctx_out].S + head_off;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = cw + 8 * nt + 2 * tq;
        *reinterpret_cast<float2*>(So + (size_t)(v0 + gq) * D + col) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(So + (size_t)(v0 + gq + 8) * D + col) = make_float2(acc[nt][2], acc[nt][3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// chunk_out: one CTA per (chunk, head, value slice), 256 threads, at least two CTAs per SM (at
// most 128 registers a thread). A CTA forms the output columns [vs * D/VS, (vs + 1) * D/VS) of
// its head; the launcher splits the value columns over VS CTAs when (chunks x heads) alone leaves
// SMs idle (a few questions over a snapshot).
//   P = lower_incl(Gamma * Q K^T),  U = Ut - W S_c^T,  O = diag(gamma) Q S_c^T + P U
// with S_c the chunk's start state: the state pass's record, or (a single-chunk sequence without
// a state pass) the snapshot's state it continues, or zero.
template <int D, int VS>
struct OutSmem {
  static constexpr int DW = D / VS;  // value columns of the slice
  static constexpr int SK = D + 8;   // f16 stride of D-wide tiles
  static constexpr int SU = DW + 8;  // f16 stride of U
  static constexpr int SP = C + 8;   // f16 stride of P
  __half Q[C * SK];
  __half K[C * SK];                  // normalised k, then U ([C][SU])
  __half W[C * SK];
  __half S[DW * SK];                 // chunk-start state rows of the slice, [v][k]
  __half P[C * SP];
  float g[C];
};

template <int D, int VS>
__global__ void __launch_bounds__(256, 2) chunk_out_kernel(const float* __restrict__ proj, int ld,
                                                        const float* __restrict__ gbuf,
                                                        const ChunkDesc* __restrict__ chunks, int H, float eps,
                                                        GdnBufs bufs, const SeqDesc* __restrict__ seqs,
                                                        const CtxDesc* __restrict__ ctxs, int layer_g, int out_fold,
                                                        f16* __restrict__ out) {
  allow_dependents();
  wait_prerequisites();
  extern __shared__ __align__(16) uint8_t smraw[];
  using SM = OutSmem<D, VS>;
  constexpr int SK = SM::SK, SU = SM::SU, SP = SM::SP, DW = SM::DW;
  constexpr int NTO = DW / 16;           // 8-column n-tiles per warp of U and O
  constexpr int PER = D / 4;
  SM& s = *reinterpret_cast<SM*>(smraw);
  const int ci = blockIdx.x, h = blockIdx.y, cs = blockIdx.z * DW;
  const ChunkDesc cd = chunks[ci];
  const int n = cd.len;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const size_t DD = (size_t)D * D;
  // this thread's quarter of row rq of q, requested first (its loads are in flight while the
  // tile copies below are issued)
  const int rq = tid >> 2, cq = (tid & 3) * PER;
  const bool okq = rq < n;
  float qv[PER];
  {
    const float* pr = proj + (size_t)(cd.row0 + (okq ? rq : 0)) * ld + h * D + cq;
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
      const float4 t = ld4(pr + i, okq);
      qv[i] = t.x; qv[i + 1] = t.y; qv[i + 2] = t.z; qv[i + 3] = t.w;
    }
  }
  for (int i = tid; i < C * (D / 8); i += 256) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < n;
    const size_t o = ((size_t)(cd.row0 + (ok ? r : 0)) * H + h) * D + c8;
    cp16(&s.K[r * SK + c8], bufs.Kn + o, ok);
    cp16(&s.W[r * SK + c8], bufs.W + o, ok);
  }
  const bool fold = cd.seq >= out_fold;
  if (!fold) {
    const f16* rec = bufs.Srec + ((size_t)ci * H + h) * DD + (size_t)cs * D;
    for (int i = tid; i < DW * (D / 8); i += 256) {
      const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
      cp16(&s.S[r * SK + c8], rec + (size_t)r * D + c8, true);
    }
  }
  cp_commit();
  if (fold) {
    const int cin = seqs[cd.seq].ctx_in;
    const float* S0 = cin >= 0 ? ctxs[cin].S + (size_t)(layer_g * H + h) * DD + (size_t)cs * D : nullptr;
    for (int i = tid; i < DW * (D / 4); i += 256) {
      const int r = i / (D / 4), c4 = (i % (D / 4)) * 4;
      const float4 v = S0 ? *reinterpret_cast<const float4*>(S0 + (size_t)r * D + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<uint2*>(&s.S[r * SK + c4]) = make_uint2(h2u(v.x, v.y), h2u(v.z, v.w));
    }
  }
  if (tid < C) s.g[tid] = tid < n ? gbuf[(size_t)(cd.row0 + tid) * H + h] : 0.f;
  // q <- q / sqrt(sum q^2 + eps) (four threads per row)
  {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) ss += qv[i] * qv[i];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = 1.0f / sqrtf(ss + eps);
#pragma unroll
    for (int i = 0; i < PER; i += 8)
      *reinterpret_cast<uint4*>(&s.Q[rq * SK + cq + i]) =
          make_uint4(h2u(qv[i] * inv, qv[i + 1] * inv), h2u(qv[i + 2] * inv, qv[i + 3] * inv),
                     h2u(qv[i + 4] * inv, qv[i + 5] * inv), h2u(qv[i + 6] * inv, qv[i + 7] * inv));
  }
  cp_wait<0>();
  __syncthreads();
  const int m0 = (warp & 3) * 16;
  // warp -> rows m0.., value columns cb .. cb + DW/2 of the slice (NTO n-tiles)
  const int cb = (warp >> 2) * (DW / 2);
  const int ta = m0 + gq, tb = m0 + gq + 8;
  // this thread's Ut values (rows ta, tb; its 2 columns of each n-tile), loaded ahead of use
  uint32_t utv[NTO][2];
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) {
    const int c = cs + cb + nt * 8 + 2 * tq;
    utv[nt][0] = ta < n ? *reinterpret_cast<const uint32_t*>(bufs.Ut + ((size_t)(cd.row0 + ta) * H + h) * D + c) : 0u;
    utv[nt][1] = tb < n ? *reinterpret_cast<const uint32_t*>(bufs.Ut + ((size_t)(cd.row0 + tb) * H + h) * D + c) : 0u;
  }
  // P = lower_incl(exp(g_t - g_s) q_t.k_s): warp -> rows m0.., key columns 32*(warp>>2) .. +31
  {
    float acc[4][4] = {};
    const int nb = (warp >> 2) * 32;
#pragma unroll
    for (int k = 0; k < D; k += 32) {
      uint32_t a0[4], a1[4];
      lda(s.Q, SK, m0, k, lane, a0);
      lda(s.Q, SK, m0, k + 16, lane, a1);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t b[4];
        ldb_nk(s.K, SK, nb + nt * 8, k, lane, b);
        mma16(acc[nt], a0, b[0], b[1]);
        mma16(acc[nt], a1, b[2], b[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = nb + nt * 8 + 2 * tq;
      const int ta = m0 + gq, tb = m0 + gq + 8;
      const float va0 = (c <= ta && ta < n) ? __expf(s.g[ta] - s.g[c]) * acc[nt][0] : 0.f;
      const float va1 = (c + 1 <= ta && ta < n) ? __expf(s.g[ta] - s.g[c + 1]) * acc[nt][1] : 0.f;
      const float vb0 = (c <= tb && tb < n) ? __expf(s.g[tb] - s.g[c]) * acc[nt][2] : 0.f;
      const float vb1 = (c + 1 <= tb && tb < n) ? __expf(s.g[tb] - s.g[c + 1]) * acc[nt][3] : 0.f;
      *reinterpret_cast<uint32_t*>(&s.P[ta * SP + c]) = h2u(va0, va1);
      *reinterpret_cast<uint32_t*>(&s.P[tb * SP + c]) = h2u(vb0, vb1);
    }
  }
  // W S^T (before Ut) and O = Q S^T over the slice's value columns
  float u[NTO][4] = {}, o[NTO][4] = {};
#pragma unroll
  for (int k = 0; k < D; k += 32) {
    uint32_t w0[4], w1[4], q0[4], q1[4];
    lda(s.W, SK, m0, k, lane, w0);
    lda(s.W, SK, m0, k + 16, lane, w1);
    lda(s.Q, SK, m0, k, lane, q0);
    lda(s.Q, SK, m0, k + 16, lane, q1);
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) {
      uint32_t b[4];
      ldb_nk(s.S, SK, cb + nt * 8, k, lane, b);
      mma16(u[nt], w0, b[0], b[1]);
      mma16(u[nt], w1, b[2], b[3]);
      mma16(o[nt], q0, b[0], b[1]);
      mma16(o[nt], q1, b[2], b[3]);
    }
  }
  {
    const float ga = __expf(s.g[ta]), gb = __expf(s.g[tb]);
#pragma unroll
    for (int nt = 0; nt < NTO; ++nt) { o[nt][0] *= ga; o[nt][1] *= ga; o[nt][2] *= gb; o[nt][3] *= gb; }
  }
  __syncthreads();   // every warp has read K (for P) before U overwrites it, and P is complete
  __half* Us = s.K;
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) {
    const int c = cb + nt * 8 + 2 * tq;
    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&utv[nt][0]));
    const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&utv[nt][1]));
    *reinterpret_cast<uint32_t*>(&Us[ta * SU + c]) = h2u(ta < n ? x.x - u[nt][0] : 0.f, ta < n ? x.y - u[nt][1] : 0.f);
    *reinterpret_cast<uint32_t*>(&Us[tb * SU + c]) = h2u(tb < n ? y.x - u[nt][2] : 0.f, tb < n ? y.y - u[nt][3] : 0.f);
  }
  __syncthreads();
  // O += P U
#pragma unroll
  for (int k = 0; k < C; k += 16) {
    uint32_t a[4];
    lda(s.P, SP, m0, k, lane, a);
#pragma unroll
    for (int nt = 0; nt < NTO; nt += 2) {
      uint32_t b[4];
      ldb_kn2(Us, SU, cb + nt * 8, k, lane, b);
      mma16(o[nt], a, b[0], b[1]);
      mma16(o[nt + 1], a, b[2], b[3]);
    }
  }
  const int HDv = H * D;
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) {
    const int c = cs + cb + nt * 8 + 2 * tq;
    if (ta < n)
      *reinterpret_cast<uint32_t*>(out + (size_t)(cd.row0 + ta) * HDv + h * D + c) = h2u(o[nt][0], o[nt][1]);
    if (tb < n)
      *reinterpret_cast<uint32_t*>(out + (size_t)(cd.row0 + tb) * HDv + h * D + c) = h2u(o[nt][2], o[nt][3]);
  }
}

}  // namespace gc

bool gdn_chunked_supported(int H, int Dk, int Dv, int ld) {
  return Dk == Dv && (Dk == 64 || Dk == 128) && H > 0 && (ld % 4) == 0;
}

size_t gdn_row_bytes(int H, int D) { return (size_t)4 * H * D * sizeof(f16); }
size_t gdn_chunk_bytes(int H, int D) { return (size_t)H * D * D * 2 * sizeof(f16) + (size_t)H * sizeof(float); }

GdnBufs gdn_bufs(void* rows, size_t R, void* per_chunk, size_t n_chunks, int H, int D) {
  GdnBufs b;
  const size_t rn = R * H * (size_t)D;
  b.Kn = (f16*)rows;
  b.W = b.Kn + rn;
  b.Ut = b.W + rn;
  b.Kp = b.Ut + rn;
  const size_t cn = n_chunks * H * (size_t)D * D;
  b.NT = (f16*)per_chunk;
  b.Srec = b.NT + cn;
  b.gam = (float*)(b.Srec + cn);
  b.rows = R;
  b.n_chunks_cap = n_chunks;
  return b;
}

template <int D, int NST>
static constexpr size_t state_smem() { return sizeof(gc::StateSmem<D, NST>) + 1024; }

template <int D>
static cudaError_t launch_state(const CUtensorMap* maps, const SeqDesc* d_seq, int n_seq, const ChunkDesc* d_chunks,
                                const CtxDesc* d_ctx, int layer_g, int H, const GdnBufs& bufs, int* d_err,
                                int num_sms, cudaStream_t st) {
  if (n_seq <= 0) return cudaSuccess;
  const dim3 grid(n_seq, H, D / gc::BV);
  if ((long)n_seq * H * (D / gc::BV) > num_sms) {   // several waves: two CTAs per SM
    CK_RET(launch_pdl(gc::chunk_state_kernel<D, 2>, grid, dim3(gc::state_threads<D>()), state_smem<D, 2>(), st,
                      maps[0], maps[1], maps[2], (const float*)bufs.gam, d_seq, d_chunks, d_ctx, layer_g, H,
                      bufs.Srec, d_err));
  } else {
    CK_RET(launch_pdl(gc::chunk_state_kernel<D, gc::NS>, grid, dim3(gc::state_threads<D>()), state_smem<D, gc::NS>(),
                      st, maps[0], maps[1], maps[2], (const float*)bufs.gam, d_seq, d_chunks, d_ctx, layer_g, H,
                      bufs.Srec, d_err));
  }
  return cudaGetLastError();
}

template <int D, int VS>
static cudaError_t launch_out(int n_chunks, int H, cudaStream_t st, const float* proj, int ld, const float* g,
                              const ChunkDesc* d_chunks, float eps, const GdnBufs& bufs, const SeqDesc* d_seq,
                              const CtxDesc* d_ctx, int layer_g, int out_fold, f16* out) {
  CK_RET(launch_pdl(gc::chunk_out_kernel<D, VS>, dim3(n_chunks, H, VS), dim3(256), sizeof(gc::OutSmem<D, VS>), st,
                    proj, ld, g, d_chunks, H, eps, bufs, d_seq, d_ctx, layer_g, out_fold, out));
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_chunked_d(const float* proj, int ld, float* gbuf, float eps, f16* out, const SeqDesc* d_seq,
                                    int n_seq, const ChunkDesc* d_chunks, int n_chunks, const CtxDesc* d_ctx,
                                    int layer_g, int H, const GdnBufs& bufs, int n_first, int fold_from, int out_fold,
                                    int* d_err, int num_sms, cudaStream_t st) {
  constexpr int VMAX = D / 32;   // most value slices of chunk_out (each slice >= 32 columns)
  static bool attr = false;
  const size_t sp = sizeof(gc::PrepSmem<D>);
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gc::chunk_prep_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if constexpr (D == 128)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gc::chunk_prep_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gc::chunk_state_kernel<D, gc::NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)state_smem<D, gc::NS>());
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
      e = cudaFuncSetAttribute(gc::chunk_out_kernel<D, VMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(gc::OutSmem<D, VMAX>));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  // every sequence a single chunk that continues a snapshot (the questions of a decide call) and
  // too few (chunk, head) pairs to fill the GPU: the right-hand side of the solve is split over
  // two CTAs per pair
  bool split_prep = false;
  if constexpr (D == 128) split_prep = out_fold == 0 && (long)n_chunks * H * 2 <= 2L * num_sms;
  if (split_prep) {
    if constexpr (D == 128)
      CK_RET(launch_pdl(gc::chunk_prep_kernel<D, true>, dim3(n_chunks, H, 2), dim3(256), sp, st, proj, ld, gbuf,
                        d_chunks, d_seq, H, eps, bufs));
  } else {
    CK_RET(launch_pdl(gc::chunk_prep_kernel<D>, dim3(n_chunks, H), dim3(256), sp, st, proj, ld, gbuf, d_chunks, d_seq,
                      H, eps, bufs));
  }
  // TMA views of the state pass's tiles: N^T [n_chunks * H * D rows, D columns] (boxes of 64
  // columns x D rows), K' and Ut [R, H, D] (64 rows of one head: 64-column swizzled boxes of K',
  // the CTA's 16 columns of Ut)
  CUtensorMap maps[3];
  {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)n_chunks * H * D};
    const uint64_t str[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, (uint32_t)D};
    const uint64_t dr[3] = {(uint64_t)D, (uint64_t)H, (uint64_t)bufs.rows};
    const uint64_t sr[2] = {(uint64_t)D * 2, (uint64_t)H * D * 2};
    const uint32_t bk[3] = {64, 1, (uint32_t)gc::C}, bu[3] = {(uint32_t)gc::BV, 1, (uint32_t)gc::C};
    if (!tensor_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, bufs.NT, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tensor_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, bufs.Kp, dr, sr, bk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tensor_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, bufs.Ut, dr, sr, bu, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  // sequences [0, n_first) run before the rest (the rest continue from their states). Sequences
  // from fold_from on are followers whose start state their prefix's state pass records;
  // sequences from out_fold on are single chunks whose start state chunk_out reads from the
  // snapshot: neither gets a state pass.
  const int split = (n_first > 0 && n_first < n_seq) ? n_first : n_seq;
  const int n1 = std::min(split, std::min(fold_from, out_fold));
  cudaError_t e = launch_state<D>(maps, d_seq, n1, d_chunks, d_ctx, layer_g, H, bufs, d_err, num_sms, st);
  if (e != cudaSuccess) return e;
  const int n2 = std::min(n_seq, out_fold) - split;
  if (split < n_seq && fold_from > split && n2 > 0) {
    e = launch_state<D>(maps, d_seq + split, n2, d_chunks, d_ctx, layer_g, H, bufs, d_err, num_sms, st);
    if (e != cudaSuccess) return e;
  }
  // value columns split over up to VMAX CTAs while (chunks x heads) CTAs leave SMs idle
  int vs = 1;
  while (vs < VMAX && (long)n_chunks * H * vs < num_sms) vs *= 2;
  if (vs == 1)
    return launch_out<D, 1>(n_chunks, H, st, proj, ld, gbuf, d_chunks, eps, bufs, d_seq, d_ctx, layer_g, out_fold, out);
  if (vs == 2)
    return launch_out<D, 2>(n_chunks, H, st, proj, ld, gbuf, d_chunks, eps, bufs, d_seq, d_ctx, layer_g, out_fold, out);
  return launch_out<D, VMAX>(n_chunks, H, st, proj, ld, gbuf, d_chunks, eps, bufs, d_seq, d_ctx, layer_g, out_fold,
                             out);
}

cudaError_t launch_gdn_chunked(const float* proj, int ld, float* gbuf, float eps, f16* out, const SeqDesc* d_seq,
                               int n_seq, const ChunkDesc* d_chunks, int n_chunks, const CtxDesc* d_ctx, int layer_g,
                               int H, int Dk, int Dv, const GdnBufs& bufs, int n_first, int fold_from, int out_fold,
                               int* d_err, int num_sms, cudaStream_t st, long* launches) {
  if (n_seq <= 0 || n_chunks <= 0) return cudaSuccess;
  if (!gdn_chunked_supported(H, Dk, Dv, ld)) return cudaErrorNotSupported;
  if (n_seq > 65535 || (size_t)n_chunks > bufs.n_chunks_cap || (size_t)n_chunks * H * Dk > 2147483647u)
    return cudaErrorInvalidValue;
  cudaError_t e = (Dk == 128)
                      ? launch_chunked_d<128>(proj, ld, gbuf, eps, out, d_seq, n_seq, d_chunks, n_chunks, d_ctx, layer_g,
                                              H, bufs, n_first, fold_from, out_fold, d_err, num_sms, st)
                      : launch_chunked_d<64>(proj, ld, gbuf, eps, out, d_seq, n_seq, d_chunks, n_chunks, d_ctx, layer_g,
                                             H, bufs, n_first, fold_from, out_fold, d_err, num_sms, st);
  if (launches) {
    const int split = (n_first > 0 && n_first < n_seq) ? n_first : n_seq;
    *launches += 2 + (std::min(split, std::min(fold_from, out_fold)) > 0 ? 1 : 0) +
                 (split < n_seq && fold_from > split && std::min(n_seq, out_fold) > split ? 1 : 0);
  }
  return e;
}

}  // namespace s1
