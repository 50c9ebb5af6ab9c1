// Causal GQA attention over packed sequences, with suffix-over-prefix continuation.
//
// A query at row i of sequence s (position pos0 + i, pos0 = P of the snapshot it continues)
// attends to every cached key of that snapshot (positions 0 .. P-1) and to its own sequence's
// keys 0 .. i; never to another sequence ("execute isolated question/option suffixes",
// System1-Omni RFC #114, section 4, "Branching" row). q head h reads kv head floor(h*Hkv/Hq).
// out = softmax(q.k / sqrt(hd)) v, online (running max / sum) softmax in fp32.
//
// Keys are addressed as one virtual array per sequence: j < P -> snapshot row j, j >= P ->
// the sequence's own row j - P. Key j has position j, query i has position P + i, so the
// causal rule is j <= P + i.
//
// flash kernel: CTA = 64 queries x one q head (4 warps x 16 rows); K/V tiles of 64 keys staged
// in shared memory by cp.async (double-buffered, 16-byte chunks XOR-swizzled by row);
// S = Q K^T and O += P V on the tensor cores (mma.sync m16n8k16 f16 -> fp32).
#include <algorithm>

#include "common.cuh"

namespace s1 {

namespace fa {

constexpr int BQ = 64, BKV = 64;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;   // src-size 0 -> zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// float at shared-memory address `saddr` of cluster CTA `rank`
__device__ __forceinline__ float ld_cluster_f32(uint32_t saddr, uint32_t rank) {
  uint32_t a;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(saddr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

// byte offset of 16-byte chunk c of row r in a tile whose rows are HD f16 wide
template <int HD>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * (HD * 2) + ((c ^ (r & 7)) << 4));
}

template <int HD>
__global__ void __launch_bounds__(128) flash_kernel(const f16* __restrict__ q, const f16* __restrict__ knew,
                                                    const f16* __restrict__ vnew, f16* __restrict__ out,
                                                    const SeqDesc* __restrict__ seqs,
                                                    const CtxDesc* __restrict__ ctxs, int layer_f, int Hq,
                                                    int Hkv, float scale_log2, int nparts) {
  allow_dependents();
  wait_prerequisites();
  constexpr int CH = HD / 8;                 // 16-byte chunks per row
  constexpr int TILE = BKV * HD * 2;         // bytes per K or V tile
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* sQ = sm;                          // BQ x HD
  uint8_t* sK = sm + BQ * HD * 2;            // 2 stages
  uint8_t* sV = sK + 2 * TILE;               // 2 stages

  const SeqDesc sd = seqs[blockIdx.z];
  // nparts CTAs (a cluster, consecutive in x) share a query tile, each taking one contiguous
  // part of its key tiles; the last (longest-key-range) query tiles go first
  const int part = (int)(blockIdx.x % nparts);
  const int q0 = ((int)(gridDim.x / nparts) - 1 - (int)(blockIdx.x / nparts)) * BQ;
  if (q0 >= sd.len) return;   // uniform over the cluster
  const int h = blockIdx.y;
  const int g = (h * Hkv) / Hq;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int P = 0;
  const f16* Kc = nullptr;
  const f16* Vc = nullptr;
  if (sd.ctx_in >= 0) {
    const CtxDesc c = ctxs[sd.ctx_in];
    P = c.P;
    const size_t plane = (size_t)c.cap * Hkv * HD;
    Kc = c.KV + (size_t)layer_f * 2 * plane + (size_t)g * HD;
    Vc = Kc + plane;
  }
  const f16* Kn = knew + ((size_t)sd.row0 * Hkv + g) * HD;
  const f16* Vn = vnew + ((size_t)sd.row0 * Hkv + g) * HD;
  const size_t kstride = (size_t)Hkv * HD;
  const int n_keys = P + min(sd.len, q0 + BQ);     // keys any query of this tile can see
  const int n_all = (n_keys + BKV - 1) / BKV;
  const int per = (n_all + nparts - 1) / nparts;
  const int t_begin = min(n_all, part * per), t_end = min(n_all, t_begin + per);

  // ---- stage Q (rows beyond len are zero)
  for (int i = tid; i < BQ * CH; i += 128) {
    const int r = i / CH, c = i % CH;
    const bool ok = q0 + r < sd.len;
    const f16* src = q + ((size_t)(sd.row0 + (ok ? q0 + r : 0)) * Hq + h) * HD + c * 8;
    cp_async16(smem_u32(sQ) + swz<HD>(r, c), src, ok);
  }
  auto load_kv = [&](int t, int stage) {
    const int j0 = t * BKV;
    for (int i = tid; i < BKV * CH; i += 128) {
      const int r = i / CH, c = i % CH;
      const int j = j0 + r;
      const bool ok = j < n_keys;
      const f16* ks;
      const f16* vs;
      if (j < P) { ks = Kc + (size_t)j * kstride; vs = Vc + (size_t)j * kstride; }
      else { const int jj = ok ? j - P : 0; ks = Kn + (size_t)jj * kstride; vs = Vn + (size_t)jj * kstride; }
      cp_async16(smem_u32(sK + stage * TILE) + swz<HD>(r, c), ks + c * 8, ok);
      cp_async16(smem_u32(sV + stage * TILE) + swz<HD>(r, c), vs + c * 8, ok);
    }
  };
  if (t_begin < t_end) load_kv(t_begin, 0);
  cp_commit();

  // Q fragments (A operand), rows 16*warp .. +15
  cp_wait<0>();
  __syncthreads();
  uint32_t qa[HD / 16][4];
  {
    const int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const int c = 2 * kk + (lane >> 4);
      ldsm_x4(smem_u32(sQ) + swz<HD>(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }
  }
  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int qi0 = q0 + warp * 16 + (lane >> 2);    // this thread's rows: qi0 and qi0 + 8
  const int lim0 = P + qi0, lim1 = P + qi0 + 8;    // last visible key index

  for (int t = t_begin; t < t_end; ++t) {
    const int stage = (t - t_begin) & 1;
    if (t + 1 < t_end) load_kv(t + 1, stage ^ 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const uint32_t kb = smem_u32(sK + stage * TILE), vb = smem_u32(sV + stage * TILE);
    // S = Q K^T  (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {       // pairs of 8-key n-tiles
        const int key = np * 16 + 8 * (lane >> 4) + (lane & 7);
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<HD>(key, c), b0, b1, b2, b3);
        mma16816(s[2 * np], qa[kk], b0, b1);
        mma16816(s[2 * np + 1], qa[kk], b2, b3);
      }
    }
    // mask + online softmax (log2 domain)
    const int j0 = t * BKV;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int jb = j0 + n * 8 + 2 * (lane & 3);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = jb + e;
        s[n][e] = (j <= lim0 && j < n_keys) ? s[n][e] * scale_log2 : -INFINITY;
        s[n][2 + e] = (j <= lim1 && j < n_keys) ? s[n][2 + e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[n][e]);
        mx1 = fmaxf(mx1, s[n][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float sc0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
    const float sc1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
    const float base0 = (mn0 == -INFINITY) ? 0.f : mn0, base1 = (mn1 == -INFINITY) ? 0.f : mn1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pa[4][4];                       // P as A fragments, one per 16-key step
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = exp2f(s[n][0] - base0), p1 = exp2f(s[n][1] - base0);
      const float p2 = exp2f(s[n][2] - base1), p3 = exp2f(s[n][3] - base1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      pa[n >> 1][(n & 1) * 2 + 0] = pack_f16(p0, p1);
      pa[n >> 1][(n & 1) * 2 + 1] = pack_f16(p2, p3);
    }
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
    rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
    rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
    l0 = l0 * sc0 + rs0;
    l1 = l1 * sc1 + rs1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) { o[i][0] *= sc0; o[i][1] *= sc0; o[i][2] *= sc1; o[i][3] *= sc1; }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < BKV / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < HD / 16; ++np) {
        const int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = 2 * np + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<HD>(key, c), b0, b1, b2, b3);
        mma16816(o[2 * np], pa[kk], b0, b1);
        mma16816(o[2 * np + 1], pa[kk], b2, b3);
      }
    }
    __syncthreads();
  }
  if (nparts > 1) {
    // publish this part's (o, m, l) in shared memory (the K/V buffers, no longer read), k-major
    // by thread; rank 0 merges the parts in rank order
    constexpr int NO = HD / 2;               // o values per thread
    float* pub = reinterpret_cast<float*>(sK);
#pragma unroll
    for (int i = 0; i < HD / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) pub[(i * 4 + e) * 128 + tid] = o[i][e];
    pub[(NO + 0) * 128 + tid] = m0;
    pub[(NO + 1) * 128 + tid] = m1;
    pub[(NO + 2) * 128 + tid] = l0;
    pub[(NO + 3) * 128 + tid] = l1;
    cluster_sync();
    if (cluster_ctarank() == 0) {
      const uint32_t base = smem_u32(pub);
      auto peer = [&](int k, int r) { return ld_cluster_f32(base + (uint32_t)((k * 128 + tid) * 4), (uint32_t)r); };
      float M0 = -INFINITY, M1 = -INFINITY;
      for (int r = 0; r < nparts; ++r) {
        M0 = fmaxf(M0, peer(NO + 0, r));
        M1 = fmaxf(M1, peer(NO + 1, r));
      }
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      for (int r = 0; r < nparts; ++r) {
        const float pm0 = peer(NO + 0, r), pm1 = peer(NO + 1, r);
        const float w0 = pm0 == -INFINITY ? 0.f : exp2f(pm0 - M0);
        const float w1 = pm1 == -INFINITY ? 0.f : exp2f(pm1 - M1);
        L0 += w0 * peer(NO + 2, r);
        L1 += w1 * peer(NO + 3, r);
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
          o[i][0] += w0 * peer(i * 4 + 0, r);
          o[i][1] += w0 * peer(i * 4 + 1, r);
          o[i][2] += w1 * peer(i * 4 + 2, r);
          o[i][3] += w1 * peer(i * 4 + 3, r);
        }
      }
      l0 = L0;
      l1 = L1;
    }
    cluster_sync();   // the peers' partials stay in place until rank 0 has read them
    if (cluster_ctarank() != 0) return;
  }
  // normalise and store rows qi0, qi0 + 8
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int col = 2 * (lane & 3);
  if (qi0 < sd.len) {
    f16* op = out + ((size_t)(sd.row0 + qi0) * Hq + h) * HD + col;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i)
      *reinterpret_cast<uint32_t*>(op + i * 8) = pack_f16(o[i][0] * inv0, o[i][1] * inv0);
  }
  if (qi0 + 8 < sd.len) {
    f16* op = out + ((size_t)(sd.row0 + qi0 + 8) * Hq + h) * HD + col;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i)
      *reinterpret_cast<uint32_t*>(op + i * 8) = pack_f16(o[i][2] * inv1, o[i][3] * inv1);
  }
}

}  // namespace fa

// Key-range parts per query tile (the cluster size): the longest key range decides.
static int attention_parts(int max_keys) {
  const int tiles = (max_keys + fa::BKV - 1) / fa::BKV;
  return tiles <= 4 ? 1 : (tiles <= 24 ? 2 : 4);
}

template <int HD>
static cudaError_t launch_flash(dim3 grid, int nparts, int smem, cudaStream_t st, const f16* q, const f16* knew,
                                const f16* vnew, f16* out, const SeqDesc* d_seq, const CtxDesc* d_ctx, int layer_f,
                                int Hq, int Hkv, float scale_log2) {
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(fa::flash_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = nparts;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, fa::flash_kernel<HD>, q, knew, vnew, out, d_seq, d_ctx, layer_f, Hq, Hkv, scale_log2,
                            nparts);
}

cudaError_t launch_attention(const f16* q, const f16* knew, const f16* vnew, f16* out,
                             const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx, int layer_f,
                             int Hq, int Hkv, int hd, int max_len, int max_keys, long work_ctas, int num_sms,
                             cudaStream_t st) {
  if (n_seq <= 0 || max_len <= 0) return cudaSuccess;
  if (n_seq > 65535) return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  // split key ranges only when the query tiles alone leave SMs idle (two CTAs fit per SM)
  const int nparts = work_ctas >= 2L * num_sms ? 1 : attention_parts(std::max(max_keys, max_len));
  dim3 grid(((max_len + fa::BQ - 1) / fa::BQ) * nparts, Hq, n_seq);
  cudaError_t e;
  if (hd == 128)
    e = launch_flash<128>(grid, nparts, fa::BQ * 128 * 2 + 4 * fa::BKV * 128 * 2, st, q, knew, vnew, out, d_seq, d_ctx,
                          layer_f, Hq, Hkv, scale_log2);
  else if (hd == 64)
    e = launch_flash<64>(grid, nparts, fa::BQ * 64 * 2 + 4 * fa::BKV * 64 * 2, st, q, knew, vnew, out, d_seq, d_ctx,
                         layer_f, Hq, Hkv, scale_log2);
  else
    return cudaErrorNotSupported;
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace s1
