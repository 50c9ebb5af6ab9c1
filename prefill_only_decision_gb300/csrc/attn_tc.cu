// Causal GQA attention with suffix-over-prefix continuation on the 5th-generation tensor cores.
//
// A query at row i of sequence s (position P + i, P = the rows of the snapshot it continues)
// attends to every cached key of that snapshot (positions 0 .. P-1) and to its own sequence's
// keys 0 .. i; never to another sequence ("execute isolated question/option suffixes",
// System1-Omni RFC #114, section 4, "Branching" row). q head h reads kv head floor(h*Hkv/Hq).
// out = softmax(q.k / sqrt(hd)) v with an online (running max / sum) softmax in fp32.
//
// One CTA per (128-query tile, q head, sequence), or per part of its key tiles when the key range
// is split over a thread-block cluster of 2 or 4 CTAs (parts merged by rank 0 over distributed
// shared memory, in rank order). Warp-specialised, 10 warps:
//   warp 0     TMA producer: the Q tile once, then K and V tiles of 128 keys (two stages), from
//              the snapshot's K/V planes (cached keys) or the call's new K/V rows (own keys);
//              the two sources never share a tile, so each tile is one box per 64 columns.
//   warp 1     TMEM allocator and MMA issuer (one thread): S = Q K^T (M 128, N 128, K hd) into
//              one of two TMEM buffers, then O += P V (M 128, N hd, K 128) into the TMEM
//              accumulator; V is read N-major (its rows are keys), P from shared memory.
//   warps 2-9  softmax, two threads per query row (one TMEM lane; warps 2-5 the first 64 keys of
//              a tile and the first half of O, warps 6-9 the rest, the row maximum and sum
//              exchanged through shared memory): mask, running max with a lazy rescale (O and l
//              are rescaled only when a row's maximum grows by more than 2^8, so P <= 256 fits
//              f16 and most tiles skip the O round trip), P as f16 into shared memory in the
//              MMA's 128-byte-swizzled K-major layout; the epilogue.
// Key masks: a cached key j is valid iff j < P (the whole snapshot is visible); an own key r is
// valid iff r <= i (causal). Rows of a tile past the sequence are computed and never stored.
// Every mbarrier wait is bounded (~1 s of %globaltimer): on expiry the kernel records an error
// code, every role leaves its loop, in-flight copies and MMAs are waited for, and TMEM is freed.
#include <algorithm>

#include "common.cuh"

namespace s1 {
namespace fat {

constexpr int BQ = 128, BKV = 128;
constexpr int NTHREADS = 320;
constexpr int ST = 2;                       // K/V stages
constexpr int TMEM_COLS = 512;              // S (2 x 128 columns) + O (hd columns)
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr int ERR_TIMEOUT = 0x301;

template <int HD>
struct Lay {
  static constexpr int Q = 0;                          // HD/64 boxes of [128 rows][128 B]
  static constexpr int TILE = BKV * HD * 2;            // one K or V tile
  static constexpr int K = Q + BQ * HD * 2;
  static constexpr int V = K + ST * TILE;
  static constexpr int P = V + ST * TILE;              // 2 boxes of [128 rows][64 keys]
  static constexpr int XCH = P + BQ * BKV * 2;         // row maxima / sums of the two halves [3][2][BQ]
  static constexpr int BAR = XCH + 3 * 2 * BQ * 4;
  // barriers and alignment slack; at least 120 KB, so that two CTAs never share an SM: each
  // allocates all 512 TMEM columns, and CTAs of one cluster wait for one another
  static constexpr int BYTES = (BAR + 256 + 1024) > 120 * 1024 ? (BAR + 256 + 1024) : 120 * 1024;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false (with the error recorded) on expiry or when another role gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* d_err) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (*abort_flag) return false;
      if (now_ns() - t0 > WAIT_NS) {
        *abort_flag = 1;
        atomicExch(d_err, ERR_TIMEOUT);
        return false;
      }
    }
  }
}
// Bounded wait that ignores the abort flag (used to drain copies and MMAs before leaving).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return;
    if ((it & 255) == 0 && now_ns() - t0 > WAIT_NS) return;
  }
}
__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma4(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle: K-major operands (8-row groups 1024 B
// apart, the leading offset unused), or N-major operands (the leading offset = the distance
// between 64-element blocks along N, the stride offset = between 8-row groups along K).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor, kind::f16: f16 A and B, fp32 D, A K-major, B K-major (b_mn = 0) or
// N-major (b_mn = 1, bit 16), N / 8 in bits 17-22, M / 16 in bits 24-28; M = 128.
__host__ __device__ constexpr uint32_t idesc(int n, int b_mn) {
  return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive TMEM columns of this thread's lane (valid after ld_wait)
__device__ __forceinline__ void tld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tst32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t h2u(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(saddr), "r"(rank));
  return a;
}
// Loads from a peer's shared memory (published before a cluster barrier, so no ordering is
// needed among the loads themselves: they issue back to back).
__device__ __forceinline__ float ld_peer(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 ld_peer4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}

// mapQ: q [R, Hq, hd] as (hd, Hq, R), box (64, 1, 128); mapKn / mapVn: new K / V [R, Hkv, hd] as
// (hd, Hkv, R), box (64, 1, 128); ctx_maps[c]: snapshot c's K/V [nF, 2, cap, Hkv, hd] as
// (hd, Hkv, cap, 2 nF), box (64, 1, 128, 1) (plane 2l = K, 2l + 1 = V of full-attention layer l).
template <int HD>
__global__ void __launch_bounds__(NTHREADS, 1)
    flash_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapKn,
                    const __grid_constant__ CUtensorMap mapVn, const CUtensorMap* __restrict__ ctx_maps,
                    f16* __restrict__ out, const SeqDesc* __restrict__ seqs, const CtxDesc* __restrict__ ctxs,
                    int layer_f, int Hq, int Hkv, float scale_log2, int nparts, int* __restrict__ d_err) {
  using L = Lay<HD>;
  constexpr int NB = HD / 64;                // 64-column boxes per row of Q, K, V
  constexpr int PSTR = HD + 4;               // floats per published row (o, m, l; 16-byte rows)
  static_assert(BQ * PSTR * 4 <= 2 * ST * L::TILE, "published partials fit the K/V stage buffers");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR);
  uint64_t* q_full = bars;
  // K and V of a stage have barriers of their own: K_i's slot is free once S_i = Q K_i^T has
  // completed, V_i's once P_i V_i has, so K_{i+ST} is requested a tile earlier than V_{i+ST}
  uint64_t* k_full = bars + 1;               // [ST]
  uint64_t* v_full = bars + 1 + ST;          // [ST]
  uint64_t* k_empty = bars + 1 + 2 * ST;     // [ST]
  uint64_t* v_empty = bars + 1 + 3 * ST;     // [ST]
  uint64_t* s_full = bars + 1 + 4 * ST;      // [2]
  uint64_t* s_empty = bars + 3 + 4 * ST;     // [2]
  uint64_t* p_full = bars + 5 + 4 * ST;
  uint64_t* o_done = bars + 6 + 4 * ST;
  uint64_t* mma_idle = bars + 7 + 4 * ST;
  uint64_t* xbar = bars + 8 + 4 * ST;        // [4 quadrants][2 tile parities + 1]: the two softmax
                                             // warps of a row quadrant meet here (2 arrivals)
  uint32_t* tmem_slot = (uint32_t*)(bars + 20 + 4 * ST);
  static_assert((20 + 4 * ST) * 8 + 6 * 4 <= 256, "barriers and counters fit their 256 bytes");
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* k_waited = (int*)(tmem_slot + 2);     // K tiles the MMA issuer saw arrive
  int* k_issued = (int*)(tmem_slot + 3);     // K tiles the producer requested
  int* v_waited = (int*)(tmem_slot + 4);     // V tiles the MMA issuer saw arrive
  int* v_issued = (int*)(tmem_slot + 5);     // V tiles the producer requested

  allow_dependents();
  wait_prerequisites();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // sequences in reverse call order: the calls list the prefixes first and the sequences that
  // continue them (whose query tiles see the most keys) after, so those start in the first wave
  const SeqDesc sd = seqs[gridDim.z - 1 - blockIdx.z];
  // x = head x key part (a cluster's parts adjacent), y = query tile: blocks go out in x order
  // first, so every head's longest query tile is handed out before any head's shorter ones
  const int part = (int)(blockIdx.x % nparts);
  const int q0 = ((int)gridDim.y - 1 - (int)blockIdx.y) * BQ;   // longest tiles first
  const int h = (int)(blockIdx.x / nparts), g = (h * Hkv) / Hq;
  // (the early exit is uniform over a cluster: its CTAs share q0)
  if (q0 >= sd.len) return;
  int P = 0;
  const CUtensorMap* cmap = nullptr;
  if (sd.ctx_in >= 0) {
    P = ctxs[sd.ctx_in].P;
    cmap = ctx_maps + sd.ctx_in;
  }
  const int ncache = (P + BKV - 1) / BKV;
  const int qend = min(sd.len, q0 + BQ);
  const int nown = (qend + BKV - 1) / BKV;
  const int total = ncache + nown;
  const int per = (total + nparts - 1) / nparts;
  const int jb = min(total, part * per), je = min(total, jb + per);
  const int n = je - jb;                     // key tiles of this CTA (0 for an empty part)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1); mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1); mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) { mbar_init(&s_full[b], 1); mbar_init(&s_empty[b], 8); }
    mbar_init(p_full, 8);
    for (int x = 0; x < 12; ++x) mbar_init(&xbar[x], 2);
    mbar_init(o_done, 1);
    mbar_init(mma_idle, 1);
    *abort_flag = 0;
    *k_waited = 0;
    *k_issued = 0;
    *v_waited = 0;
    *v_issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0 && n > 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapQ)) : "memory");
      mbar_expect_tx(q_full, BQ * HD * 2);
#pragma unroll
      for (int b = 0; b < NB; ++b) tma3(sm + L::Q + b * BQ * 128, &mapQ, q_full, 64 * b, h, sd.row0 + q0);
      for (int i = 0; i < n; ++i) {
        const int s = i % ST, j = jb + i;
        const int rnew = sd.row0 + (j - ncache) * BKV;   // (own keys) the tile's first packed row
        if (!mbar_wait(&k_empty[s], ((i / ST) & 1) ^ 1, abort_flag, d_err)) break;
        mbar_expect_tx(&k_full[s], L::TILE);
        *k_issued = i + 1;
        uint8_t* kd = sm + L::K + s * L::TILE;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (j < ncache) tma4(kd + b * BKV * 128, cmap, &k_full[s], 64 * b, g, j * BKV, 2 * layer_f);
          else tma3(kd + b * BKV * 128, &mapKn, &k_full[s], 64 * b, g, rnew);
        }
        if (!mbar_wait(&v_empty[s], ((i / ST) & 1) ^ 1, abort_flag, d_err)) break;
        mbar_expect_tx(&v_full[s], L::TILE);
        *v_issued = i + 1;
        uint8_t* vd = sm + L::V + s * L::TILE;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (j < ncache) tma4(vd + b * BKV * 128, cmap, &v_full[s], 64 * b, g, j * BKV, 2 * layer_f + 1);
          else tma3(vd + b * BKV * 128, &mapVn, &v_full[s], 64 * b, g, rnew);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t ID_S = idesc(BKV, 0), ID_O = idesc(HD, 1);
      const uint32_t tO = tmem + 256;
      bool ok = mbar_wait(q_full, 0, abort_flag, d_err);
      auto issue_s = [&](int i) -> bool {   // S_i = Q K_i^T into S buffer i & 1
        const int s = i % ST, b = i & 1;
        if (!mbar_wait(&k_full[s], (i / ST) & 1, abort_flag, d_err)) return false;
        *k_waited = i + 1;
        if (!mbar_wait(&s_empty[b], ((i >> 1) & 1) ^ 1, abort_flag, d_err)) return false;
        fence_after();
        const uint32_t qa = smem_u32(sm + L::Q), ka = smem_u32(sm + L::K + s * L::TILE);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * (128 * 128) + (kk & 3) * 32);
          mma(tmem + b * 128, desc_sw128(qa + off, 16), desc_sw128(ka + off, 16), ID_S, kk > 0 ? 1u : 0u);
        }
        commit(&s_full[b]);
        commit(&k_empty[s]);
        return true;
      };
      auto issue_pv = [&](int i) -> bool {   // O += P_i V_i
        const int s = i % ST;
        if (!mbar_wait(p_full, i & 1, abort_flag, d_err)) return false;
        if (!mbar_wait(&v_full[s], (i / ST) & 1, abort_flag, d_err)) return false;
        *v_waited = i + 1;
        fence_after();
        const uint32_t pa = smem_u32(sm + L::P), va = smem_u32(sm + L::V + s * L::TILE);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const uint32_t poff = (uint32_t)((kk >> 2) * (128 * 128) + (kk & 3) * 32);
          const uint32_t voff = (uint32_t)(kk * 16 * 128);   // 16 key rows
          mma(tO, desc_sw128(pa + poff, 16), desc_sw128(va + voff, BKV * 128), ID_O, (i > 0 || kk > 0) ? 1u : 0u);
        }
        commit(o_done);
        commit(&v_empty[s]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 0; i < n && ok; ++i) {
        if (i + 1 < n) ok = issue_s(i + 1);
        if (ok) ok = issue_pv(i);
      }
      commit(mma_idle);                      // arrives once every MMA issued above has completed
      mbar_drain(mma_idle, 0);
    }
  } else {
    // ---- softmax warps: two threads per query row r (TMEM lane r), warps 2-5 the row's first
    // half of the scores, warps 6-9 its second half. Waits are agreed on by the whole warp, so
    // the warp-collective TMEM accesses below never diverge.
    auto wwait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, d_err) ? 1 : 0) != 0;
    };
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;        // 0: key columns 0..63 of a tile, 1: 64..127
    const int r = quad * 32 + lane;
    const int qi = q0 + r;                   // query index within the sequence
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256 + (uint32_t)(half * (HD / 2));   // this half's O columns
    uint8_t* prow = sm + L::P + half * (BQ * 128) + r * 128;   // this row in P's box `half`
    float* xch = reinterpret_cast<float*>(sm + L::XCH);         // [3][2 halves][BQ]
    // the two warps of a row quadrant meet on an mbarrier of two arrivals (a bounded wait)
    auto pair_meet = [&](int slot, uint32_t parity) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[quad * 3 + slot]);
      return wwait(&xbar[quad * 3 + slot], parity);
    };
    constexpr int HB = BKV / 2;              // scores per thread and tile
    float m = -INFINITY, l = 0.f;            // l: this half's share of the row sum
    bool ok = n > 0;
    for (int i = 0; i < n && ok; ++i) {
      const int j = jb + i, b = i & 1;
      if (!wwait(&s_full[b], (i >> 1) & 1)) { ok = false; break; }
      fence_after();
      float sv[HB];
      {
        uint32_t u[HB];   // the half row's two 32-column loads in flight together
#pragma unroll
        for (int c = 0; c < HB; c += 32) tld32(tmem + lane_off + b * 128 + half * HB + c, u + c);
        ld_wait();
#pragma unroll
        for (int c = 0; c < HB; ++c) sv[c] = __uint_as_float(u[c]);
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[b]);
      // mask and scale (log2 domain)
      const bool cache = j < ncache;
      const int kbase = (cache ? j * BKV : (j - ncache) * BKV) + half * HB;
      const int klim = cache ? P - 1 : qi;   // last visible key of this tile's source
      float mx = -INFINITY;
      if (kbase + HB - 1 <= klim) {          // every key of this half tile is visible to this row
#pragma unroll
        for (int c = 0; c < HB; ++c) {
          sv[c] *= scale_log2;
          mx = fmaxf(mx, sv[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HB; ++c) {
          sv[c] = (kbase + c <= klim) ? sv[c] * scale_log2 : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      }
      // the row's maximum over both halves (a buffer per tile parity: the next tile writes the
      // other one, and the tile after that comes only after both threads passed the next barrier)
      xch[(b * 2 + half) * BQ + r] = mx;
      if (!pair_meet(b, (i >> 1) & 1)) { ok = false; break; }
      mx = fmaxf(mx, xch[(b * 2 + (half ^ 1)) * BQ + r]);
      // lazy rescale: move the reference maximum only when it grows by more than 8 (2^8); both
      // halves of a row see the same maxima, so they take the same decisions
      float alpha = 1.f;
      if (mx > m + 8.f) {
        alpha = (m == -INFINITY) ? 1.f : exp2f(m - mx);
        m = mx;
      }
      const float base = (m == -INFINITY) ? 0.f : m;
      float rs = 0.f;
      // the previous tile's P V has finished: P may be rewritten and O rescaled
      if (i > 0 && !wwait(o_done, (i - 1) & 1)) { ok = false; break; }
      fence_after();
      if (__any_sync(0xffffffffu, alpha != 1.f) && i > 0) {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < HD / 2; c += 32) {
          tld32(tO + c, u);
          ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
          tst32(tO + c, u);
        }
        st_wait();
      }
      l *= alpha;
#pragma unroll
      for (int c8 = 0; c8 < HB / 8; ++c8) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = exp2f(sv[c8 * 8 + e] - base);
          rs += p[e];
        }
        // 16-byte chunk c8 of the row in box `half`: chunk c8 ^ (r % 8)
        uint4 v = make_uint4(h2u(p[0], p[1]), h2u(p[2], p[3]), h2u(p[4], p[5]), h2u(p[6], p[7]));
        *reinterpret_cast<uint4*>(prow + (((c8 ^ (r & 7))) << 4)) = v;
      }
      l += rs;
      fence_async_smem();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ---- epilogue: O row / l (merged over the cluster's parts first); each thread its half of
    // the O columns, the row sum over both halves
    constexpr int HO = HD / 2;
    float o[HO];
    if (ok && n > 0) {
      ok = wwait(o_done, (n - 1) & 1);
      fence_after();
      if (ok) {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < HO; c += 32) {
          tld32(tO + c, u);
          ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[c + e] = __uint_as_float(u[e]);
        }
      }
    }
    if (!ok || n == 0) {
#pragma unroll
      for (int c = 0; c < HO; ++c) o[c] = 0.f;
      if (!ok) { m = -INFINITY; l = 0.f; }
    }
    // the row sum over both halves (every exit of the loop above falls through to here)
    xch[(2 * 2 + half) * BQ + r] = l;
    if (pair_meet(2, 0)) l += xch[(2 * 2 + (half ^ 1)) * BQ + r];
    else ok = false;
    if (nparts > 1) {
      // publish (o, m, l) in the K/V stage buffers (no longer read once every tile was consumed),
      // one row of PSTR floats per query row
      float* pub = reinterpret_cast<float*>(sm + L::K) + r * PSTR;
#pragma unroll
      for (int c = 0; c < HO; c += 4)
        *reinterpret_cast<float4*>(pub + half * HO + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
      if (half == 0) {
        pub[HD] = m;
        pub[HD + 1] = l;
      }
    }
    if (nparts == 1) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (qi < sd.len && ok) {
        f16* op = out + ((size_t)(sd.row0 + qi) * Hq + h) * HD + half * HO;
#pragma unroll
        for (int c = 0; c < HO; c += 8)
          *reinterpret_cast<uint4*>(op + c) =
              make_uint4(h2u(o[c] * inv, o[c + 1] * inv), h2u(o[c + 2] * inv, o[c + 3] * inv),
                         h2u(o[c + 4] * inv, o[c + 5] * inv), h2u(o[c + 6] * inv, o[c + 7] * inv));
      }
    }
  }
  __syncthreads();
  // the producer's copies that the MMA issuer never waited for (an aborted call) land before exit
  if (threadIdx.x == 0 && *abort_flag) {
    for (int i = *k_waited; i < *k_issued; ++i) mbar_drain(&k_full[i % ST], (i / ST) & 1);
    for (int i = *v_waited; i < *v_issued; ++i) mbar_drain(&v_full[i % ST], (i / ST) & 1);
  }
  if (nparts > 1) {
    cluster_sync();
    // every CTA of the cluster merges HD / nparts of the output columns of all 128 rows, from
    // the parts in rank order; the two threads of a row take alternate 16-column groups
    if (warp >= 2) {
      const int half = (warp - 2) >> 2;
      const int r = (warp & 3) * 32 + lane, qi = q0 + r;
      const uint32_t rank = cluster_rank();
      const uint32_t row = smem_u32(sm + L::K) + (uint32_t)(r * PSTR * 4);
      float pm[4], pl[4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
        if (p < nparts) {
          const uint32_t a = peer_addr(row, (uint32_t)p);
          pm[p] = ld_peer(a + HD * 4);
          pl[p] = ld_peer(a + (HD + 1) * 4);
        }
      float M = -INFINITY;
#pragma unroll
      for (int p = 0; p < 4; ++p)
        if (p < nparts) M = fmaxf(M, pm[p]);
      float Lsum = 0.f, w[4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
        if (p < nparts) {
          w[p] = pm[p] == -INFINITY ? 0.f : exp2f(pm[p] - M);
          Lsum += w[p] * pl[p];
        }
      const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
      const int cw = HD / nparts, c0 = (int)rank * cw;   // this CTA's columns (a multiple of 16)
      for (int cb = 16 * half; cb < cw; cb += 32) {
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          if (p >= nparts) break;
          const uint32_t a = peer_addr(row, (uint32_t)p) + (uint32_t)((c0 + cb) * 4);
          float4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = ld_peer4(a + 16 * q);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[4 * q] += w[p] * v[q].x;
            acc[4 * q + 1] += w[p] * v[q].y;
            acc[4 * q + 2] += w[p] * v[q].z;
            acc[4 * q + 3] += w[p] * v[q].w;
          }
        }
        if (qi < sd.len && !*abort_flag) {
          f16* op = out + ((size_t)(sd.row0 + qi) * Hq + h) * HD + c0 + cb;
          reinterpret_cast<uint4*>(op)[0] =
              make_uint4(h2u(acc[0] * inv, acc[1] * inv), h2u(acc[2] * inv, acc[3] * inv),
                         h2u(acc[4] * inv, acc[5] * inv), h2u(acc[6] * inv, acc[7] * inv));
          reinterpret_cast<uint4*>(op)[1] =
              make_uint4(h2u(acc[8] * inv, acc[9] * inv), h2u(acc[10] * inv, acc[11] * inv),
                         h2u(acc[12] * inv, acc[13] * inv), h2u(acc[14] * inv, acc[15] * inv));
        }
      }
    }
    cluster_sync();   // every CTA's partials stay in place until all of the cluster has read them
  }
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

}  // namespace fat

// Key-range parts per query tile (the cluster size): the longest key range decides.
static int parts_for(int max_keys) {
  const int tiles = (max_keys + fat::BKV - 1) / fat::BKV;
  return tiles <= 2 ? 1 : (tiles <= 8 ? 2 : 4);
}

bool attention_tc_supported(int hd) { return hd == 64 || hd == 128; }

size_t attention_ctx_map_bytes() { return sizeof(CUtensorMap); }

// The map covers the P cached rows of each plane (rows past P read as zeros, never as the
// unwritten capacity behind them); planes are cap rows apart.
bool attention_ctx_map(void* map_out, const f16* kv, int n_fa_layers, int P, int cap, int Hkv, int hd) {
  const uint64_t dims[4] = {(uint64_t)hd, (uint64_t)Hkv, (uint64_t)std::max(P, 1), (uint64_t)2 * n_fa_layers};
  const uint64_t str[3] = {(uint64_t)hd * 2, (uint64_t)Hkv * hd * 2, (uint64_t)cap * Hkv * hd * 2};
  const uint32_t box[4] = {64, 1, (uint32_t)fat::BKV, 1};
  return tensor_map(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, kv, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int HD>
static cudaError_t launch_tc(dim3 grid, int nparts, cudaStream_t st, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, const CUtensorMap* ctx_maps, f16* out, const SeqDesc* d_seq,
                             const CtxDesc* d_ctx, int layer_f, int Hq, int Hkv, float scale_log2, int* d_err) {
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(fat::flash_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fat::Lay<HD>::BYTES);
    if (e != cudaSuccess) return e;
    set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(fat::NTHREADS);
  cfg.dynamicSmemBytes = fat::Lay<HD>::BYTES;
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
  return cudaLaunchKernelEx(&cfg, fat::flash_tc_kernel<HD>, mq, mk, mv, ctx_maps, out, d_seq, d_ctx, layer_f, Hq,
                            Hkv, scale_log2, nparts, d_err);
}

cudaError_t launch_attention_tc(const f16* q, const f16* knew, const f16* vnew, f16* out, int R,
                                const SeqDesc* d_seq, int n_seq, const CtxDesc* d_ctx, const void* d_ctx_maps,
                                int layer_f, int Hq, int Hkv, int hd, int max_len, int max_keys, long work_ctas,
                                int num_sms, int* d_err, cudaStream_t st) {
  if (n_seq <= 0 || max_len <= 0 || R <= 0) return cudaSuccess;
  if (n_seq > 65535 || (max_len + fat::BQ - 1) / fat::BQ > 65535 || !attention_tc_supported(hd))
    return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  {
    const uint64_t dq[3] = {(uint64_t)hd, (uint64_t)Hq, (uint64_t)R};
    const uint64_t sq[2] = {(uint64_t)hd * 2, (uint64_t)Hq * hd * 2};
    const uint64_t dk[3] = {(uint64_t)hd, (uint64_t)Hkv, (uint64_t)R};
    const uint64_t sk[2] = {(uint64_t)hd * 2, (uint64_t)Hkv * hd * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!tensor_map(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, q, dq, sq, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tensor_map(&mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, knew, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tensor_map(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vnew, dk, sk, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  // split key ranges over a cluster only when the query tiles alone leave SMs idle
  // key ranges split over up to parts_for() CTAs while the split still fits one wave (one CTA
  // per SM: a second wave would double the time of the whole launch)
  int nparts = 1;
  if (work_ctas < num_sms) {
    const int want = parts_for(std::max(max_keys, max_len));
    while (nparts < want && work_ctas * (nparts * 2) <= num_sms) nparts *= 2;
  }
  const dim3 grid(Hq * nparts, (max_len + fat::BQ - 1) / fat::BQ, n_seq);
  const CUtensorMap* cm = reinterpret_cast<const CUtensorMap*>(d_ctx_maps);
  cudaError_t e = hd == 128 ? launch_tc<128>(grid, nparts, st, mq, mk, mv, cm, out, d_seq, d_ctx, layer_f, Hq, Hkv,
                                             scale_log2, d_err)
                            : launch_tc<64>(grid, nparts, st, mq, mk, mv, cm, out, d_seq, d_ctx, layer_f, Hq, Hkv,
                                            scale_log2, d_err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace s1
