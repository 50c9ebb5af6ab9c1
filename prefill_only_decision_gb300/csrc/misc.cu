// Small kernels of the path: embedding gather, RMSNorm, RoPE + KV split,
// decision readout, load-time LoRA merge and the rotary table.
#include "common.cuh"

namespace s1 {

// ---- embedding rows: x[r] = E[id] (fp32), or a given embedding row ---------------------
// row_src[r] >= 0: token id; row_src[r] < 0: row (-1 - row_src[r]) of `embeds`.
// E is the model's f16 copy of the tied embedding; given rows are the caller's bf16.
__global__ void embed_kernel(const f16* __restrict__ E, const int* __restrict__ row_src,
                             const bf16* __restrict__ embeds, float* __restrict__ x, int d) {
  allow_dependents();
  const int r = blockIdx.x;
  const int s = row_src[r];
  float* dst = x + (size_t)r * d;
  if (s >= 0) {
    const f16* src = E + (size_t)s * d;
    for (int i = threadIdx.x * 2; i < d; i += blockDim.x * 2)
      *reinterpret_cast<float2*>(dst + i) = __half22float2(*reinterpret_cast<const __half2*>(src + i));
  } else {
    const bf16* src = embeds + (size_t)(-1 - s) * d;
    for (int i = threadIdx.x * 2; i < d; i += blockDim.x * 2)
      *reinterpret_cast<float2*>(dst + i) = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i));
  }
}

cudaError_t launch_embed(const f16* E, const int* row_src, const bf16* embeds, float* x, int R, int d,
                         cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  embed_kernel<<<R, 256, 0, st>>>(E, row_src, embeds, x, d);
  return cudaGetLastError();
}

// ---- RMSNorm: out = f16(x / sqrt(mean(x^2) + eps) * w) ---------------------------------
// One warp per row, the row held in registers (one read of x), 8 rows per block; the block
// stages w in shared memory while its rows load, so no global round trip follows the reduction.
// (x, the previous kernel's output, carries no __restrict__: with code ahead of the wait, its
// loads must not be treated as invariant and moved above it.)
template <int NV>   // float4 per lane: d = 128 * NV
__global__ void __launch_bounds__(256) rmsnorm_warp_kernel(const float* x, const float* __restrict__ w,
                                                           f16* __restrict__ out, int R, int d, float eps) {
  allow_dependents();
  __shared__ float4 ws[32 * NV];
  const float4* wr = reinterpret_cast<const float4*>(w);
  for (int i = threadIdx.x; i < 32 * NV; i += 256) ws[i] = wr[i];   // w does not depend on earlier kernels
  wait_prerequisites();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  float4 v[NV];
  float ss = 0.f;
  if (r < R) {
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)r * d);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      v[i] = xr[lane + 32 * i];
      ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
  }
  __syncthreads();   // ws complete (every thread reaches this, rows past R included)
  if (r >= R) return;
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  uint2* o = reinterpret_cast<uint2*>(out + (size_t)r * d);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const float4 g = ws[lane + 32 * i];
    __half2 a = __floats2half2_rn(v[i].x * inv * g.x, v[i].y * inv * g.y);
    __half2 b = __floats2half2_rn(v[i].z * inv * g.z, v[i].w * inv * g.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    o[lane + 32 * i] = u;
  }
}

// General width (d % 4 == 0): one block of norm_row_threads(d) threads per row, two passes.
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ w,
                               f16* __restrict__ out, int d, float eps) {
  allow_dependents();
  wait_prerequisites();
  __shared__ float red[32];
  const int r = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)r * d);
  float ss = 0.f;
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    float4 v = xr[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  const float4* wr = reinterpret_cast<const float4*>(w);
  __half2* o2 = reinterpret_cast<__half2*>(out + (size_t)r * d);
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    float4 v = xr[i], g = wr[i];
    o2[2 * i] = __floats2half2_rn(v.x * inv * g.x, v.y * inv * g.y);
    o2[2 * i + 1] = __floats2half2_rn(v.z * inv * g.z, v.w * inv * g.w);
  }
}

cudaError_t launch_rmsnorm(const float* x, const float* w, f16* out, int R, int d, float eps,
                           cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  const int blocks = (R + 7) / 8;
  // few rows (questions over a snapshot): a block per row spreads them over more SMs
  if (R <= 512 && d % 4 == 0) {
    CK_RET(launch_pdl(rmsnorm_kernel, dim3(R), dim3(norm_row_threads(d)), 0, st, x, w, out, d, eps));
    return cudaGetLastError();
  }
  switch (d) {
    case 256: CK_RET(launch_pdl(rmsnorm_warp_kernel<2>, dim3(blocks), dim3(256), 0, st, x, w, out, R, d, eps)); break;
    case 1024: CK_RET(launch_pdl(rmsnorm_warp_kernel<8>, dim3(blocks), dim3(256), 0, st, x, w, out, R, d, eps)); break;
    case 2560: CK_RET(launch_pdl(rmsnorm_warp_kernel<20>, dim3(blocks), dim3(256), 0, st, x, w, out, R, d, eps)); break;
    case 5120: CK_RET(launch_pdl(rmsnorm_warp_kernel<40>, dim3(blocks), dim3(256), 0, st, x, w, out, R, d, eps)); break;
    default: CK_RET(launch_pdl(rmsnorm_kernel, dim3(R), dim3(norm_row_threads(d)), 0, st, x, w, out, d, eps)); break;
  }
  return cudaGetLastError();
}

// ---- RoPE (rotate-half over the whole head) + split of the fused q|k|v projection -------
// proj row r: [q (Hq*hd) | k (Hkv*hd) | v (Hkv*hd)] fp32. Writes q, k_new, v_new (f16) at
// packed row r and, for sequences that own a snapshot, K/V into its cache at row = position.
// Grid (row, item block): one thread per item, items = the (Hq + Hkv) * hd/8 runs of four
// adjacent rotated elements of q and k (i .. i+3 with partners i + hd/2 .. i + hd/2 + 3), then the
// Hkv * hd/4 runs of four v values (16-byte loads, 8-byte stores, one round trip to memory per
// thread, so that a few rows still spread over the whole GPU).
__global__ void rope_split_kernel(const float* __restrict__ proj, int ld, const float2* __restrict__ tab,
                                  const int* __restrict__ row_seq, const SeqDesc* __restrict__ seqs,
                                  const CtxDesc* __restrict__ ctxs, int layer_f, f16* __restrict__ q,
                                  f16* __restrict__ knew, f16* __restrict__ vnew, int Hq, int Hkv,
                                  int hd) {
  allow_dependents();
  wait_prerequisites();
  const int r = blockIdx.x;
  const int half = hd / 2, eighth = hd / 8;
  const int nq = Hq * eighth, nk = Hkv * eighth;
  const int t = blockIdx.y * blockDim.x + threadIdx.x;
  if (t >= nq + nk + Hkv * eighth * 2) return;
  const float* pr = proj + (size_t)r * ld;
  const SeqDesc sd = seqs[row_seq[r]];
  const int pos = sd.pos0 + (r - sd.row0);
  f16* kc = nullptr;
  f16* vc = nullptr;
  if (sd.ctx_out >= 0) {
    const CtxDesc c = ctxs[sd.ctx_out];
    const size_t plane = (size_t)c.cap * Hkv * hd;
    kc = c.KV + (size_t)layer_f * 2 * plane + (size_t)pos * Hkv * hd;
    vc = kc + plane;
  }
  if (t < nq + nk) {
    // four adjacent elements i .. i+3 of the first half of a q or k head and their partners
    // i + hd/2 .. i + hd/2 + 3
    const bool isq = t < nq;
    const int tt = isq ? t : t - nq;
    const int h = tt / eighth, i = 4 * (tt % eighth);
    const float* src = pr + (isq ? 0 : Hq * hd) + h * hd;
    const float4 x1 = *reinterpret_cast<const float4*>(src + i);
    const float4 x2 = *reinterpret_cast<const float4*>(src + i + half);
    const float4 c01 = *reinterpret_cast<const float4*>(tab + (size_t)pos * half + i);       // (cos, sin) of i, i+1
    const float4 c23 = *reinterpret_cast<const float4*>(tab + (size_t)pos * half + i + 2);   // of i+2, i+3
    const __half2 a0 = __floats2half2_rn(x1.x * c01.x - x2.x * c01.y, x1.y * c01.z - x2.y * c01.w);
    const __half2 a1 = __floats2half2_rn(x1.z * c23.x - x2.z * c23.y, x1.w * c23.z - x2.w * c23.w);
    const __half2 b0 = __floats2half2_rn(x2.x * c01.x + x1.x * c01.y, x2.y * c01.z + x1.y * c01.w);
    const __half2 b1 = __floats2half2_rn(x2.z * c23.x + x1.z * c23.y, x2.w * c23.z + x1.w * c23.w);
    uint2 y1, y2;
    y1.x = *reinterpret_cast<const uint32_t*>(&a0); y1.y = *reinterpret_cast<const uint32_t*>(&a1);
    y2.x = *reinterpret_cast<const uint32_t*>(&b0); y2.y = *reinterpret_cast<const uint32_t*>(&b1);
    f16* dst = isq ? q + (size_t)r * Hq * hd : knew + (size_t)r * Hkv * hd;
    *reinterpret_cast<uint2*>(dst + h * hd + i) = y1;
    *reinterpret_cast<uint2*>(dst + h * hd + i + half) = y2;
    if (!isq && kc) {
      *reinterpret_cast<uint2*>(kc + h * hd + i) = y1;
      *reinterpret_cast<uint2*>(kc + h * hd + i + half) = y2;
    }
  } else {
    const int tv = 4 * (t - (nq + nk));
    const float4 x = *reinterpret_cast<const float4*>(pr + (Hq + Hkv) * hd + tv);
    const __half2 v0 = __floats2half2_rn(x.x, x.y), v1 = __floats2half2_rn(x.z, x.w);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&v0); v.y = *reinterpret_cast<const uint32_t*>(&v1);
    *reinterpret_cast<uint2*>(vnew + (size_t)r * Hkv * hd + tv) = v;
    if (vc) *reinterpret_cast<uint2*>(vc + tv) = v;
  }
}

cudaError_t launch_rope_split(const float* proj, int ld, const float2* rope_tab, const int* row_seq,
                              const SeqDesc* d_seq, const CtxDesc* d_ctx, int layer_f, f16* q,
                              f16* knew, f16* vnew, int R, int Hq, int Hkv, int hd,
                              cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  if (hd % 8 || ld % 4) return cudaErrorInvalidValue;
  const int items = (Hq + Hkv) * (hd / 8) + Hkv * (hd / 4);
  const dim3 grid(R, (items + 127) / 128);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  CK_RET(launch_pdl(rope_split_kernel, grid, dim3(128), 0, st, proj, ld, rope_tab, row_seq, d_seq, d_ctx, layer_f,
                    q, knew, vnew, Hq, Hkv, hd));
  return cudaGetLastError();
}

// cos/sin table: tab[pos*half + i] = (cos, sin)(pos * theta^(-2i/hd)), evaluated in double.
__global__ void rope_table_kernel(float2* tab, int max_pos, int hd, double theta) {
  const int half = hd / 2;
  const size_t n = (size_t)max_pos * half;
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n; t += (size_t)gridDim.x * blockDim.x) {
    const int pos = (int)(t / half), i = (int)(t % half);
    const double inv = pow(theta, -2.0 * i / (double)hd);
    double s, c;
    sincos((double)pos * inv, &s, &c);
    tab[t] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float2* tab, int max_pos, int hd, double theta, cudaStream_t st) {
  rope_table_kernel<<<1024, 256, 0, st>>>(tab, max_pos, hd, theta);
  return cudaGetLastError();
}

// ---- decision readout -----------------------------------------------------------------
// One block per question: final RMSNorm of its last row, tied-embedding logits over its
// option ids (fp32), softmax, argmax, expected level, yes probability and confidences.
// (x, the residual stream, is the previous kernels' output and is read only after the wait: it
// carries no __restrict__, so its loads are not treated as invariant and cannot move above the
// wait)
__global__ void readout_kernel(const float* x, const float* __restrict__ fnorm,
                               const f16* __restrict__ E, int d, float eps,
                               const int* __restrict__ q_row, const int* __restrict__ q_type,
                               const int* __restrict__ opt_off, const int* __restrict__ opt_ids,
                               float* __restrict__ probs, float* __restrict__ stats,
                               float* __restrict__ hidden, float* __restrict__ hn_out,
                               float* __restrict__ z_out) {
  extern __shared__ float sm[];
  float* hn = sm;            // [d]
  float* z = sm + d;         // [n]
  __shared__ float red[32];
  allow_dependents();
  const int j = blockIdx.x;
  const int row = q_row[j];
  const int o0 = opt_off[j], n = opt_off[j + 1] - o0;
  // the option rows of the tied embedding do not depend on earlier kernels: ask L2 for them
  // while the last layer finishes
  for (int i = threadIdx.x; i < n * (d / 64); i += blockDim.x) {
    const f16* e = E + (size_t)opt_ids[o0 + i / (d / 64)] * d + (i % (d / 64)) * 64;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(e));
  }
  wait_prerequisites();
  const float* h = x + (size_t)row * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = h[i];
    ss += v * v;
    if (hidden) hidden[(size_t)j * d + i] = v;
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)d + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    hn[i] = h[i] * inv * fnorm[i];
    if (hn_out) hn_out[(size_t)j * d + i] = hn[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int m = w; m < n; m += nw) {
    const f16* e = E + (size_t)opt_ids[o0 + m] * d;
    float acc = 0.f;
    if (d % 256 == 0) {   // eight halves per lane and load
      for (int i = 8 * lane; i < d; i += 256) {
        const uint4 u = *reinterpret_cast<const uint4*>(e + i);
        const __half2* e2 = reinterpret_cast<const __half2*>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(e2[k]);
          acc += hn[i + 2 * k] * f.x + hn[i + 2 * k + 1] * f.y;
        }
      }
    } else {
      for (int i = lane; i < d; i += 32) acc += hn[i] * h2f(e[i]);
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      z[m] = acc;
      if (z_out) z_out[o0 + m] = acc;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float mx = -INFINITY;
    int am = 0;
    for (int m = 0; m < n; ++m) if (z[m] > mx) { mx = z[m]; am = m; }
    float se = 0.f;
    for (int m = 0; m < n; ++m) se += expf(z[m] - mx);
    const float lse = logf(se);
    float ent = 0.f, ex = 0.f, p2 = 0.f;
    for (int m = 0; m < n; ++m) {
      const float lp = z[m] - mx - lse;
      const float p = expf(lp);
      probs[o0 + m] = p;
      if (p > 0.f) ent -= p * lp;
      ex += (float)m * p;
      if (m != am && p > p2) p2 = p;
    }
    const float pmax = expf(-lse);
    const float econf = (n == 1) ? 1.f : 1.f - ent / logf((float)n);
    float* s = stats + (size_t)j * 8;
    s[0] = (float)am;
    s[1] = ex;
    s[2] = expf(z[0] - mx - lse);
    s[3] = pmax;
    s[4] = (q_type[j] == 2) ? pmax : econf;
    s[5] = econf;
    s[6] = pmax - p2;
    s[7] = (float)n;
  }
}

cudaError_t launch_readout(const float* x, const float* final_norm, const f16* E, int d, float eps,
                           const int* q_row, const int* q_type, const int* opt_off,
                           const int* opt_ids, int n_q, float* probs, float* stats, float* hidden,
                           int max_opts, float* hn_out, float* z_out, cudaStream_t st) {
  if (n_q <= 0) return cudaSuccess;
  const size_t smem = (size_t)(d + max_opts) * sizeof(float);
  if (smem > 48 * 1024) {
    CK_RET(cudaFuncSetAttribute(readout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  }
  CK_RET(launch_pdl(readout_kernel, dim3(n_q), dim3(256), smem, st, x, final_norm, E, d, eps, q_row, q_type, opt_off,
                    opt_ids, probs, stats, hidden, hn_out, z_out));
  return cudaGetLastError();
}

// ---- load-time: W' = W + scale * B A (fp32 accumulate, one f16 rounding) -----------------
// dst row mapping: plain (dst_row0 + o), or SwiGLU interleave: the gate (half 0) / up
// (half 1) row o lands at 32*(o/16) + 16*half + o%16 of the packed [2F, in] matrix.
__device__ __forceinline__ float ld_any(const void* p, int is_bf16, size_t i) {
  return is_bf16 ? __bfloat162float(reinterpret_cast<const bf16*>(p)[i])
                 : reinterpret_cast<const float*>(p)[i];
}

__global__ void merge_lora_kernel(const void* __restrict__ W, int w_bf16, const void* __restrict__ A,
                                  const void* __restrict__ B, int ab_bf16, int rank, float scale,
                                  int out_f, int in_f, f16* __restrict__ dst, int dst_row0,
                                  int interleave, int half) {
  const int o = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= in_f) return;
  float acc = ld_any(W, w_bf16, (size_t)o * in_f + i);
  if (rank > 0) {
    float t = 0.f;
    for (int r = 0; r < rank; ++r)
      t = fmaf(ld_any(B, ab_bf16, (size_t)o * rank + r), ld_any(A, ab_bf16, (size_t)r * in_f + i), t);
    acc = fmaf(scale, t, acc);
  }
  const int drow = interleave ? (32 * (o / 16) + 16 * half + (o % 16)) : (dst_row0 + o);
  dst[(size_t)drow * in_f + i] = __float2half_rn(acc);
}

cudaError_t launch_merge_lora(const void* W, int w_is_bf16, const void* A, const void* B,
                              int ab_is_bf16, int rank, float scale, int out_f, int in_f,
                              f16* dst, int dst_row0, int interleave_swiglu, int swiglu_half,
                              int swiglu_F, float* tmpA, float* tmpB, cudaStream_t st) {
  (void)swiglu_F; (void)tmpA; (void)tmpB;
  if (interleave_swiglu && out_f > 65535) return cudaErrorNotSupported;
  // grid.y is limited to 65535 rows per launch: split tall matrices (plain mapping only).
  for (int o0 = 0; o0 < out_f; o0 += 65535) {
    const int rows = (out_f - o0) < 65535 ? (out_f - o0) : 65535;
    dim3 grid((in_f + 255) / 256, rows);
    const void* Wc = (const char*)W + (size_t)o0 * in_f * (w_is_bf16 ? 2 : 4);
    const void* Bc = B ? (const void*)((const char*)B + (size_t)o0 * rank * (ab_is_bf16 ? 2 : 4)) : nullptr;
    merge_lora_kernel<<<grid, 256, 0, st>>>(Wc, w_is_bf16, A, Bc, ab_is_bf16, rank, scale, rows, in_f,
                                            dst, dst_row0 + o0, interleave_swiglu, swiglu_half);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

__global__ void to_f32_kernel(const void* __restrict__ src, int is_bf16, float* __restrict__ dst, size_t n) {
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n; t += (size_t)gridDim.x * blockDim.x)
    dst[t] = ld_any(src, is_bf16, t);
}

cudaError_t launch_to_f32(const void* src, int is_bf16, float* dst, size_t n, cudaStream_t st) {
  to_f32_kernel<<<256, 256, 0, st>>>(src, is_bf16, dst, n);
  return cudaGetLastError();
}

}  // namespace s1
