// Gated delta rule (Gated DeltaNet) kernels.
//
// Per layer and head, with q, k L2-normalised:
//   alpha_t = exp(-softplus(a_t)), beta_t = sigmoid(b_t)
//   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t
// (Yang, Kautz & Hatamizadeh, "Gated Delta Networks", 2024). The state is kept in fp32, as
// the pages' snapshot does ("FP32 Gated DeltaNet recurrent state", System1-Omni RFC #114,
// section 5). Every row i of S evolves independently given (k, alpha, beta):
//   s_i <- alpha s_i + beta (v_i - alpha s_i.k) k,    o_i = alpha s_i.q + u_i (k.q)
// with s_i the previous row and u_i = beta (v_i - alpha s_i.k). The scan therefore splits
// the value dimension across CTAs: grid (sequence, head, Dv / 16).
#include "common.cuh"

namespace s1 {

// q, k <- x / sqrt(sum x^2 + eps) per head (in place); loga = -softplus(a); beta = sigmoid(b).
// proj row: [q (H*Dk) | k (H*Dk) | v (H*Dv) | a (H) | b (H)].
__global__ void gdn_prep_kernel(float* __restrict__ proj, int ld, float* __restrict__ loga,
                                float* __restrict__ beta, int H, int Dk, int Dv, float eps) {
  allow_dependents();
  wait_prerequisites();
  const int r = blockIdx.x;
  float* pr = proj + (size_t)r * ld;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int j = w; j < 2 * H; j += nw) {            // j < H: q head j; else k head j-H
    float* x = pr + (size_t)j * Dk;
    float ss = 0.f;
    for (int i = lane; i < Dk; i += 32) ss += x[i] * x[i];
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss + eps);
    // stored rounded to TF32 (10-bit mantissa): every later product of q and k runs on TF32
    // tensor-core inputs, so the rounding happens once here instead of at each use
    for (int i = lane; i < Dk; i += 32) {
      uint32_t r;
      asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x[i] * inv));
      x[i] = __uint_as_float(r);
    }
  }
  const float* ab = pr + 2 * H * Dk + H * Dv;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float a = ab[h], b = ab[H + h];
    const float sp = fmaxf(a, 0.f) + log1pf(expf(-fabsf(a)));   // softplus(a)
    loga[(size_t)r * H + h] = -sp;
    beta[(size_t)r * H + h] = 1.f / (1.f + expf(-b));
  }
}

cudaError_t launch_gdn_prep(float* proj, int ld, float* loga, float* beta, int R, int H, int Dk,
                            int Dv, float eps, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  CK_RET(launch_pdl(gdn_prep_kernel, dim3(R), dim3(256), 0, st, proj, ld, loga, beta, H, Dk, Dv, eps));
  return cudaGetLastError();
}

// Token-by-token scan. Block = 4 warps x 4 state rows = 16 rows of one head; a lane holds
// E = Dk/32 consecutive columns of each of its warp's rows. Next-token operands are loaded
// one step ahead (they do not depend on the state).
template <int DK>
__global__ void __launch_bounds__(128) gdn_scan_token_kernel(
    const float* __restrict__ proj, int ld, const float* __restrict__ loga,
    const float* __restrict__ beta, f16* __restrict__ out, const SeqDesc* __restrict__ seqs,
    const CtxDesc* __restrict__ ctxs, int layer_g, int H, int Dv) {
  allow_dependents();
  wait_prerequisites();
  constexpr int E = DK / 32;
  const int sq = blockIdx.x, h = blockIdx.y;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int rbase = blockIdx.z * 16 + w * 4;       // first of this warp's 4 value rows
  const SeqDesc sd = seqs[sq];
  const size_t head_off = (size_t)(layer_g * H + h) * Dv * DK;
  float s[4][E];
  if (sd.ctx_in >= 0) {
    const float* S0 = ctxs[sd.ctx_in].S + head_off;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) s[r][e] = S0[(size_t)(rbase + r) * DK + lane * E + e];
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) s[r][e] = 0.f;
  }
  const int HDk = H * DK;
  const float* qb = proj + h * DK + lane * E;
  const float* kb = proj + HDk + h * DK + lane * E;
  const float* vb = proj + 2 * HDk + h * Dv + rbase;
  float kn[E], qn[E], vn[4], lan = 0.f, ben = 0.f;
  auto load = [&](int row) {
    const size_t o = (size_t)row * ld;
#pragma unroll
    for (int e = 0; e < E; ++e) { kn[e] = kb[o + e]; qn[e] = qb[o + e]; }
#pragma unroll
    for (int r = 0; r < 4; ++r) vn[r] = vb[o + r];
    lan = loga[(size_t)row * H + h];
    ben = beta[(size_t)row * H + h];
  };
  if (sd.len > 0) load(sd.row0);
  for (int t = 0; t < sd.len; ++t) {
    const int row = sd.row0 + t;
    float k[E], q[E], v[4];
#pragma unroll
    for (int e = 0; e < E; ++e) { k[e] = kn[e]; q[e] = qn[e]; }
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = vn[r];
    const float al = __expf(lan), be = ben;
    if (t + 1 < sd.len) load(row + 1);
    float dk[4], dq[4], kq = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) kq = fmaf(k[e], q[e], kq);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      dk[r] = 0.f; dq[r] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) { dk[r] = fmaf(s[r][e], k[e], dk[r]); dq[r] = fmaf(s[r][e], q[e], dq[r]); }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kq += __shfl_xor_sync(0xffffffffu, kq, o);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        dk[r] += __shfl_xor_sync(0xffffffffu, dk[r], o);
        dq[r] += __shfl_xor_sync(0xffffffffu, dq[r], o);
      }
    }
    float ov[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float u = be * (v[r] - al * dk[r]);
#pragma unroll
      for (int e = 0; e < E; ++e) s[r][e] = fmaf(al, s[r][e], u * k[e]);
      ov[r] = fmaf(al, dq[r], u * kq);
    }
    if (lane < 4) {
      float val = ov[0];
#pragma unroll
      for (int r = 1; r < 4; ++r) if (lane == r) val = ov[r];
      out[(size_t)row * H * Dv + h * Dv + rbase + lane] = f2h(val);
    }
  }
  if (sd.ctx_out >= 0) {
    float* So = ctxs[sd.ctx_out].S + head_off;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) So[(size_t)(rbase + r) * DK + lane * E + e] = s[r][e];
  }
}

cudaError_t launch_gdn_scan(const float* proj, int ld, const float* loga, const float* beta,
                            f16* out, const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx,
                            int layer_g, int H, int Dk, int Dv, cudaStream_t st) {
  if (n_seq <= 0) return cudaSuccess;
  if (Dk != Dv || (Dv % 16) != 0) return cudaErrorNotSupported;
  dim3 grid(n_seq, H, Dv / 16);
  if (Dk == 128)
    CK_RET(launch_pdl(gdn_scan_token_kernel<128>, grid, dim3(128), 0, st, proj, ld, loga, beta, out, d_seq, d_ctx, layer_g, H, Dv));
  else if (Dk == 64)
    CK_RET(launch_pdl(gdn_scan_token_kernel<64>, grid, dim3(128), 0, st, proj, ld, loga, beta, out, d_seq, d_ctx, layer_g, H, Dv));
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

}  // namespace s1
