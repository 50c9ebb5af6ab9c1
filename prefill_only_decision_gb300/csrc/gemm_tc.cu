// Tensor-core GEMM for sm_103a: TMA -> shared memory -> tcgen05.mma -> TMEM -> epilogue.
//
//   Y = epi(X[M,K] . W[N,K]^T), f16 operands (both K-major), fp32 accumulation in TMEM.
//
// Persistent, warp-specialised CTA of 6 warps, one CTA per SM:
//   warp 0       TMA producer: 128 x 64 A tile and BN x 64 B tile per stage (128-byte swizzle)
//   warp 1       TMEM allocator and MMA issuer (one thread): 4 x tcgen05.mma (K = 16) per stage
//   warps 2..5   epilogue: tcgen05.ld of the 128 x BN accumulator (one row per thread),
//                fused epilogue (fp32 store or residual add-reduction by TMA from swizzled
//                shared-memory boxes; f16 / SwiGLU stores from registers; split-K partials)
// The accumulator is double-buffered in TMEM (2 x 256 columns) so the epilogue of one tile
// overlaps the main loop of the next. Work units are (m tile, split, n tile) with the m tile
// fastest, so CTAs running at the same time read the same weight tile (L2 reuse). When the
// tile count cannot fill the SMs, K is split and a reduction kernel applies the epilogue in a
// fixed order (deterministic). A CTA-pair variant (tcgen05.mma.cta_group::2, 256-row tiles,
// each CTA loading its own half of the weight tile) is the other candidate; the planner and a
// per-shape autotuner choose among them. No load is multicast across a cluster. Launches use
// programmatic dependent launch.
//
// Every mbarrier wait is bounded (~1 s of %globaltimer); on expiry the kernel records an
// error code in the caller's error word and every role leaves its loop, so no launch can
// hang the GPU.
#include <cuda.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.cuh"

namespace s1 {

namespace tc {

constexpr int BM = 128, BK = 64;
constexpr int NUM_THREADS = 192;
constexpr int PF = 8;   // weight tiles are prefetched into L2 this many k blocks ahead
constexpr uint64_t WAIT_NS = 1000000000ull;   // bounded wait: 1 s
constexpr int ERR_TIMEOUT_FULL = 0x101, ERR_TIMEOUT_EMPTY = 0x102, ERR_TIMEOUT_TFULL = 0x103,
              ERR_TIMEOUT_TEMPTY = 0x104;

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
// Bounded wait. Returns false (and records `code`) if the phase does not complete in time or
// another role of this CTA has already given up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* d_err, int code) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if ((++it & 255) == 0) {
      if (*abort_flag) return false;
      if (now_ns() - t0 > WAIT_NS) {
        *abort_flag = 1;
        atomicExch(d_err, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Hint: bring a box of the tensor into L2 ahead of its TMA load (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
// Hint: bring `bytes` (multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2_bytes(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: f16 A/B (format code 0 in bits 7-9 and 10-12), fp32 D
// (bits 4-5 = 1), both K-major, N / 8 in bits 17-22, M / 16 in bits 24-28; M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_f16(int bn) {
  return (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// Issue one 32-lane x 16-column TMEM load; the values are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Keeps the compiler from moving uses of a TMEM-loaded value above tmem_wait_ld().
__device__ __forceinline__ void reg_fence(float& x) { asm volatile("" : "+f"(x)); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}


// ---- CTA-pair (cta_group::2) forms ----------------------------------------------------------
// Address of the same shared-memory variable in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// TMA load into this CTA's shared memory that completes its bytes on an mbarrier of either CTA
// of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// D[256 x N] (+)= A[256 x 16] . B[N x 16]^T over the CTA pair: A rows 0..127 and B rows
// 0..N/2-1 from the issuing CTA's shared memory, the rest from the peer's at the same offsets;
// D rows 0..127 land in the issuing CTA's TMEM, rows 128..255 in the peer's.
__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive (when the pair's earlier MMAs issued by this thread complete) on `bar` in both CTAs.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a barrier that the peer CTA also arrives on.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  int* d_err, int code) {
  const uint64_t t0 = now_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_cluster(bar, parity)) return true;
    if ((++it & 255) == 0) {
      if (*abort_flag) return false;
      if (now_ns() - t0 > WAIT_NS) {
        *abort_flag = 1;
        atomicExch(d_err, code);
        return false;
      }
    }
  }
}

// Instruction descriptor for the pair: M = 256.
__host__ __device__ constexpr uint32_t idesc_f16_pair(int bn) {
  return (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}


// ---- epilogue bulk stores ----------------------------------------------------------------------
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// box of the output tensor at (x, y) <- shared memory (rows outside the tensor are not written)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
// box of the output tensor at (x, y) += shared memory, element by element in L2
__device__ __forceinline__ void tma_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Epilogue staging: two 2 KB boxes (32 rows x 64 bytes) per epilogue warp.
constexpr int STG_BYTES = 4 * 2 * 2048;
// Shared memory left for pipeline stages: the opt-in maximum less staging, barriers and alignment.
constexpr int STAGE_BUDGET = 232448 - STG_BYTES - 1024 - 256;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = STAGE_BUDGET / STAGE_BYTES > 8 ? 8 : STAGE_BUDGET / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + STG_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};


// TMEM columns the pair kernel allocates (in both CTAs of the pair, collectively).
constexpr int PAIR_TMEM_COLS = 512;

// Per-CTA stage of the pair kernel: 128 A rows and half of the BN B rows.
template <int BN>
struct Cfg2 {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / 2) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = STAGE_BUDGET / STAGE_BYTES > 8 ? 8 : STAGE_BUDGET / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + STG_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

struct Params {
  int M, N, K;
  int m_tiles, n_tiles, splits, kb_per_split, kb_total;
  int m_groups;     // m work groups: m tiles (single-CTA kernel) or 256-row pair tiles
  int units;        // work units: m_groups x splits x n_tiles
  int epi;          // epilogue; EPI_PARTIAL = write fp32 partials to ws
  void* out;
  int ldo;
  float* ws;        // split-K partials [splits, m_tiles*BM, N]
  int* d_err;
};
constexpr int EPI_PARTIAL = 100;

// Epilogue of one epilogue warp's 32 accumulator rows of a tile: TMEM -> registers (up to four
// 16-column loads in flight per wait). fp32 outputs then go through a 32 x 16 box in shared
// memory (one 64-byte row per lane, swizzled like the output map) to one TMA bulk store per box,
// or a TMA add-reduction into the fp32 residual stream for EPI_RESADD (each output element has
// exactly one writer, so the sum is the plain fp32 x + acc); a lane's row of a store box is
// 64 bytes, where a direct store from registers would write 16-byte pieces of 32 rows. f16
// outputs (32 contiguous bytes per row and chunk) are stored from registers. Two staging boxes per
// warp alternate; a box is rewritten only after the store issued from it two boxes earlier has
// read it. m0 = the warp's first row of the product, y0 = its row in the output map (m0, or
// m0 + split x padded rows for split-K partials), n0 = the tile's first column, `nst` = this
// warp's running count of issued boxes. Warps whose rows all lie past M store nothing: rows past
// the end of a padded cluster's last tile would otherwise land in the next split's partials.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const Params& p, const CUtensorMap* mapO, uint32_t tbase, int m0, int y0,
                                              int n0, uint8_t* stg, int lane, int& nst) {
  if (m0 >= p.M) return;
  auto acquire = [&]() -> uint8_t* {
    if (nst >= 2) {
      if (lane == 0) bulk_wait_read1();
      __syncwarp();
    }
    return stg + (nst & 1) * 2048;
  };
  auto issue = [&](uint8_t* box, int x) {
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (p.epi == EPI_RESADD) tma_add_2d(mapO, box, x, y0);
      else tma_store_2d(mapO, box, x, y0);
      bulk_commit();
    }
    ++nst;
  };
  // 16-byte chunk c of this lane's row in a 64-byte swizzled row (the output map's 64-byte swizzle)
  auto chunk64 = [&](uint8_t* box, int c) { return reinterpret_cast<uint4*>(box + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)); };
  float lmx = -INFINITY, lsum = 0.f;   // EPI_LSE: running max and sum of exp over the row's columns
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 64) {
    const int nc = (BN - c0) < 64 ? (BN - c0) / 16 : 4;   // 16-column chunks in this group
    float v[4][16];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nc) tmem_ld16_async(tbase + c0 + 16 * j, v[j]);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 16; ++i) reg_fence(v[j][i]);
    const int m = m0 + lane;   // this lane's output row (f16 outputs: stored from registers)
    if (p.epi == EPI_SWIGLU) {
      // chunk pairs (gate, up): tile columns [32b, 32b+16) gate, [32b+16, 32b+32) up; each row's
      // 16 outputs are 32 contiguous bytes (one full sector)
#pragma unroll
      for (int j = 0; j + 1 < 4; j += 2) {
        if (m < p.M && j + 1 < nc && n0 + c0 + 16 * j < p.N) {
          f16* o = reinterpret_cast<f16*>(p.out) + (size_t)m * p.ldo + (n0 + c0 + 16 * j) / 2;
          __align__(16) f16 r[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = f2h(silu_f(v[j][i]) * v[j + 1][i]);
          reinterpret_cast<uint4*>(o)[0] = reinterpret_cast<uint4*>(r)[0];
          reinterpret_cast<uint4*>(o)[1] = reinterpret_cast<uint4*>(r)[1];
        }
      }
    } else if (p.epi == EPI_HALF) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + c0 + 16 * j;
        if (m >= p.M || j >= nc || n >= p.N) continue;
        __align__(16) f16 r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = f2h(v[j][i]);
        uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<f16*>(p.out) + (size_t)m * p.ldo + n);
        o[0] = reinterpret_cast<uint4*>(r)[0];
        o[1] = reinterpret_cast<uint4*>(r)[1];
      }
    } else if (p.epi == EPI_LSE) {
      // N is a multiple of 32, so a chunk that starts before N is whole
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j >= nc || n0 + c0 + 16 * j >= p.N) continue;
        float cm = v[j][0];
#pragma unroll
        for (int i = 1; i < 16; ++i) cm = fmaxf(cm, v[j][i]);
        const float nm = fmaxf(lmx, cm);
        float add = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) add += __expf(v[j][i] - nm);
        lsum = lsum * __expf(lmx - nm) + add;
        lmx = nm;
      }
    } else if (p.epi == EPI_PARTIAL) {
      // split-K partials: plain stores, summed by splitk_reduce_kernel
      const size_t yr = (size_t)(y0 + lane);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + c0 + 16 * j;
        if (j >= nc || n >= p.N) continue;
        float4* o = reinterpret_cast<float4*>(p.ws + yr * p.N + n);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = make_float4(v[j][4 * i], v[j][4 * i + 1], v[j][4 * i + 2], v[j][4 * i + 3]);
      }
    } else {   // fp32 outputs: staged boxes, TMA store or add-reduction
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + c0 + 16 * j;
        if (j >= nc || n >= p.N) continue;
        uint8_t* box = acquire();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *chunk64(box, c) = make_uint4(__float_as_uint(v[j][4 * c]), __float_as_uint(v[j][4 * c + 1]),
                                        __float_as_uint(v[j][4 * c + 2]), __float_as_uint(v[j][4 * c + 3]));
        issue(box, n);
      }
    }
  }
  if (p.epi == EPI_LSE && m0 + lane < p.M)
    reinterpret_cast<float2*>(p.out)[(size_t)(n0 / BN) * p.ldo + m0 + lane] = make_float2(lmx, lsum);
}

// One CTA per SM, each loading its own A and B tiles; CTAs that run at the same time work on
// consecutive m tiles of the same n tile, so a weight tile is read from DRAM once and served to
// the others from L2.
template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapO, Params p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint8_t* stg_all = smem + C::STAGES * C::STAGE_BYTES;          // epilogue staging (1024-aligned)
  uint64_t* bars = (uint64_t*)(stg_all + STG_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = (uint32_t*)(tempty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = blockIdx.x, ncl = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], 4); }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = *tmem_slot;
  allow_dependents();
  // The weights do not depend on earlier kernels: while the kernel producing this GEMM's
  // activations may still be running, the first unit's weight tiles are requested into the
  // pipeline's stages (their A tiles follow after the wait) and the next ones into L2.
  int early = 0;   // stages of the first unit whose weight tile is already requested
  if (warp == 0 && lane == 0 && cid < p.units) {
    const int u = cid;
    const int mg = u % p.m_groups, rest = u / p.m_groups, sp = rest % p.splits, nt = rest / p.splits;
    const int kb0 = sp * p.kb_per_split, kb1 = min(p.kb_total, kb0 + p.kb_per_split);
    early = min(C::STAGES, kb1 - kb0);
    for (int i = 0; i < early; ++i) {
      mbar_expect_tx(&full[i], C::STAGE_BYTES);
      tma_load_2d(sB + i * C::B_BYTES, &mapB, &full[i], (kb0 + i) * BK, nt * BN);
    }
    if (mg == 0)
      for (int kb = kb0 + early; kb < min(kb1, kb0 + early + PF); ++kb) tma_prefetch_l2(&mapB, kb * BK, nt * BN);
  }
  wait_prerequisites();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cid; u < p.units && ok; u += ncl) {
        const int mg = u % p.m_groups;
        const int rest = u / p.m_groups;
        const int sp = rest % p.splits;
        const int nt = rest / p.splits;
        const int mt = mg;
        const int kb0 = sp * p.kb_per_split;
        const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
        // the weight tile is fetched from DRAM into L2 PF blocks ahead (only the first m tile
        // of each n tile prefetches; the others run alongside it)
        const int brow = nt * BN;
        const bool pf = mg == 0;
        if (pf)
          for (int kb = kb0; kb < min(kb1, kb0 + PF); ++kb) tma_prefetch_l2(&mapB, kb * BK, brow);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (pf && kb + PF < kb1) tma_prefetch_l2(&mapB, (kb + PF) * BK, brow);
          if (u == cid && kb - kb0 < early) {
            // (a fresh stage whose weight tile and byte count were set before the wait)
            tma_load_2d(sA + stage * C::A_BYTES, &mapA, &full[stage], kb * BK, mt * BM);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.d_err, ERR_TIMEOUT_EMPTY)) { ok = false; break; }
            mbar_expect_tx(&full[stage], C::STAGE_BYTES);
            tma_load_2d(sA + stage * C::A_BYTES, &mapA, &full[stage], kb * BK, mt * BM);
            tma_load_2d(sB + stage * C::B_BYTES, &mapB, &full[stage], kb * BK, brow);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // drain: every stage this CTA filled has been released by its MMAs before the CTA exits
      for (int i = 0; i < C::STAGES && ok; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.d_err, ERR_TIMEOUT_EMPTY)) break;
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int u = cid; u < p.units && ok; u += ncl, ++it) {
        const int rest = u / p.m_groups;
        const int sp = rest % p.splits;
        const int kb0 = sp * p.kb_per_split;
        const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
        const int buf = it & 1;
        if (!mbar_wait(&tempty[buf], ((it >> 1) & 1) ^ 1, abort_flag, p.d_err, ERR_TIMEOUT_TEMPTY)) { ok = false; break; }
        fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * 256);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.d_err, ERR_TIMEOUT_FULL)) { ok = false; break; }
          fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            mma_f16(tmem_d, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                     (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (ok) mma_commit(&tfull[buf]);
      }
    }
  } else {
    // epilogue warps 2..5: TMEM lane quadrant = warp % 4
    const int q = warp & 3;
    uint8_t* stg = stg_all + (warp - 2) * 4096;
    int nst = 0;
    int it = 0;
    for (int u = cid; u < p.units; u += ncl, ++it) {
      const int mg = u % p.m_groups;
      const int rest = u / p.m_groups;
      const int sp = rest % p.splits;
      const int nt = rest / p.splits;
      const int mt = mg;
      const int buf = it & 1;
      if (!mbar_wait(&tfull[buf], (it >> 1) & 1, abort_flag, p.d_err, ERR_TIMEOUT_TFULL)) break;
      fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 256);
      const int m0 = mt * BM + q * 32;
      epilogue_tile<BN>(p, &mapO, tbase, m0, (p.epi == EPI_PARTIAL ? sp * p.m_tiles * BM : 0) + m0, nt * BN, stg,
                        lane, nst);
      fence_before();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
    if (lane == 0) bulk_wait_all();   // this warp's stores have completed
  }
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512));
  }
}


// CTA-pair variant: a cluster of two CTAs computes a 256 x BN tile with tcgen05.mma.cta_group::2.
// Each CTA stages its own 128 A rows and one half of the B tile, so a stage costs each SM
// 16 KB + BN x 64 B of shared memory and of L2-to-SM traffic for 128 x BN x 64 of MMA work (the
// single-CTA kernel moves 16 KB + BN x 128 B for the same work): deeper pipelines and less
// traffic per FLOP. The even CTA of the pair issues the MMAs and owns the barriers that gate
// them: both CTAs' TMA loads complete on its `full` barriers, and both CTAs' epilogue warps
// release a TMEM buffer on its `tempty` barriers. Its MMA commits arrive on both CTAs' `empty`
// and `tfull` barriers. Work units are (m pair tile, split, n tile), m fastest.
template <int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                     const __grid_constant__ CUtensorMap mapO, Params p) {
  using C = Cfg2<BN>;
  static_assert((BN / 2) % 8 == 0 && BN % 16 == 0 && BN <= 256, "pair tile width");
  constexpr int BUFCOLS = BN <= 128 ? 128 : 256;          // TMEM columns per accumulator buffer
  constexpr int NBUF = PAIR_TMEM_COLS / BUFCOLS;            // accumulator buffers (1, 2 or 4)
  static_assert(NBUF >= 1 && NBUF <= 4, "TMEM buffers");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint8_t* stg_all = smem + C::STAGES * C::STAGE_BYTES;          // epilogue staging (1024-aligned)
  uint64_t* bars = (uint64_t*)(stg_all + STG_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = tfull + NBUF;
  uint32_t* tmem_slot = (uint32_t*)(tempty + NBUF);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();           // 0 = MMA issuer, 1 = peer
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < NBUF; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], 8); }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapB)) : "memory");
  }
  if (warp == 1) {   // one warp of each CTA: the pair allocates the same columns in both TMEMs
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(PAIR_TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers are initialised before any cross-CTA signal
  fence_after();
  const uint32_t tmem_base = *tmem_slot;
  allow_dependents();
  if (warp == 0 && lane == 0 && cid < p.units) {
    const int u = cid;
    const int mg = u % p.m_groups, rest = u / p.m_groups, sp = rest % p.splits, nt = rest / p.splits;
    if (mg == 0) {
      const int kb0 = sp * p.kb_per_split, kb1 = min(p.kb_total, kb0 + p.kb_per_split);
      for (int kb = kb0; kb < min(kb1, kb0 + PF); ++kb)
        tma_prefetch_l2(&mapB, kb * BK, nt * BN + (int)crank * (BN / 2));
    }
  }
  wait_prerequisites();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);   // issuer's full barriers
      for (int u = cid; u < p.units && ok; u += ncl) {
        const int mg = u % p.m_groups;
        const int rest = u / p.m_groups;
        const int sp = rest % p.splits;
        const int nt = rest / p.splits;
        const int arow = mg * (2 * BM) + (int)crank * BM;
        const int brow = nt * BN + (int)crank * (BN / 2);
        const int kb0 = sp * p.kb_per_split;
        const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
        const bool pf = mg == 0;
        if (pf)
          for (int kb = kb0; kb < min(kb1, kb0 + PF); ++kb) tma_prefetch_l2(&mapB, kb * BK, brow);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (pf && kb + PF < kb1) tma_prefetch_l2(&mapB, (kb + PF) * BK, brow);
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.d_err, ERR_TIMEOUT_EMPTY)) { ok = false; break; }
          if (crank == 0) mbar_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
          const uint32_t fb = full0 + (uint32_t)(stage * 8);
          tma_load_2d_pair(sA + stage * C::A_BYTES, &mapA, fb, kb * BK, arow);
          tma_load_2d_pair(sB + stage * C::B_BYTES, &mapB, fb, kb * BK, brow);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // drain: the issuer's releases of this CTA's stages have all arrived
      for (int i = 0; i < C::STAGES && ok; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.d_err, ERR_TIMEOUT_EMPTY)) break;
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && crank == 0) {
      constexpr uint32_t idesc = idesc_f16_pair(BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int u = cid; u < p.units && ok; u += ncl, ++it) {
        const int rest = u / p.m_groups;
        const int sp = rest % p.splits;
        const int kb0 = sp * p.kb_per_split;
        const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
        const int buf = it % NBUF, use = it / NBUF;
        if (!mbar_wait_cluster(&tempty[buf], (use & 1) ^ 1, abort_flag, p.d_err, ERR_TIMEOUT_TEMPTY)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * BUFCOLS);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.d_err, ERR_TIMEOUT_FULL)) { ok = false; break; }
          fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16_pair(tmem_d, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                          (kb > kb0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(&empty[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (ok) mma_commit_pair(&tfull[buf]);
      }
    }
  } else {
    const int q = warp & 3;
    uint8_t* stg = stg_all + (warp - 2) * 4096;
    int nst = 0;
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
    int it = 0;
    for (int u = cid; u < p.units; u += ncl, ++it) {
      const int mg = u % p.m_groups;
      const int rest = u / p.m_groups;
      const int sp = rest % p.splits;
      const int nt = rest / p.splits;
      const int buf = it % NBUF, use = it / NBUF;
      if (!mbar_wait(&tfull[buf], use & 1, abort_flag, p.d_err, ERR_TIMEOUT_TFULL)) break;
      fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BUFCOLS);
      const int m0 = mg * (2 * BM) + (int)crank * BM + q * 32;
      epilogue_tile<BN>(p, &mapO, tbase, m0, (p.epi == EPI_PARTIAL ? sp * p.m_tiles * BM : 0) + m0, nt * BN, stg,
                        lane, nst);
      fence_before();
      if (lane == 0) mbar_arrive_remote(tempty0 + (uint32_t)(buf * 8));
    }
    if (lane == 0) bulk_wait_all();   // this warp's stores have completed
  }
  __syncthreads();
  cluster_sync_all();   // neither CTA leaves while the other may still signal or read it
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(PAIR_TMEM_COLS));
  }
}

// Sum over the splits of one float4 of the partials, in split order; the loads of up to four
// splits are issued before their sums, so a row waits for one round trip to memory, not one per
// split.
__device__ __forceinline__ float4 sum_splits(const float* ws, int splits, size_t split_stride, size_t off) {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < splits; s0 += 4) {
    float4 p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (s0 + j < splits) p[j] = *reinterpret_cast<const float4*>(ws + (size_t)(s0 + j) * split_stride + off);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (s0 + j < splits) { a.x += p[j].x; a.y += p[j].y; a.z += p[j].z; a.w += p[j].w; }
  }
  return a;
}

// Sum of the split-K partials in split order, then the epilogue.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int splits, int Mpad, int M, int N, int epi,
                                     void* __restrict__ out, int ldo) {
  allow_dependents();
  wait_prerequisites();
  const int cols = (epi == EPI_SWIGLU) ? N / 2 : N;
  const size_t total = (size_t)M * (cols / 4);
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < total; t += (size_t)gridDim.x * blockDim.x) {
    const int m = (int)(t / (cols / 4));
    const int c = (int)(t % (cols / 4)) * 4;
    if (epi == EPI_SWIGLU) {
      // output column c..c+3 -> gate column 32*(c/16) + c%16, up = gate + 16
      const int gcol = 32 * (c / 16) + (c % 16);
      float4 g = make_float4(0, 0, 0, 0), u = make_float4(0, 0, 0, 0);
      for (int s = 0; s < splits; ++s) {
        const float* rp = ws + ((size_t)s * Mpad + m) * N;
        const float4 a = *reinterpret_cast<const float4*>(rp + gcol);
        const float4 b = *reinterpret_cast<const float4*>(rp + gcol + 16);
        g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
        u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
      }
      f16* o = reinterpret_cast<f16*>(out) + (size_t)m * ldo + c;
      o[0] = f2h(silu_f(g.x) * u.x); o[1] = f2h(silu_f(g.y) * u.y);
      o[2] = f2h(silu_f(g.z) * u.z); o[3] = f2h(silu_f(g.w) * u.w);
    } else {
      const float4 a = sum_splits(ws, splits, (size_t)Mpad * N, (size_t)m * N + c);
      if (epi == EPI_F32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)m * ldo + c) = a;
      } else if (epi == EPI_RESADD) {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)m * ldo + c);
        float4 x = *o;
        x.x += a.x; x.y += a.y; x.z += a.z; x.w += a.w;
        *o = x;
      } else {
        f16* o = reinterpret_cast<f16*>(out) + (size_t)m * ldo + c;
        o[0] = f2h(a.x); o[1] = f2h(a.y); o[2] = f2h(a.z); o[3] = f2h(a.w);
      }
    }
  }
}

// Split-K reduction of a residual-add GEMM with the RMSNorm that follows it: one block of
// norm_row_threads(N) threads per row sums the partials in split order, adds them to the
// residual row and writes it back, then writes the row normalised. Per element and per thread the sums run in the same order as
// splitk_reduce_kernel followed by the block-per-row RMSNorm, so the results are the same bits.
__global__ void __launch_bounds__(1024) splitk_resadd_norm_kernel(const float* __restrict__ ws, int splits, int Mpad,
                                                                 int N, float* __restrict__ x, int ldx,
                                                                 const float* __restrict__ w, f16* __restrict__ xn,
                                                                 float eps) {
  allow_dependents();
  wait_prerequisites();
  __shared__ float red[32];
  const int m = blockIdx.x;
  float4* xr = reinterpret_cast<float4*>(x + (size_t)m * ldx);
  float ss = 0.f;
  for (int i = threadIdx.x; i < N / 4; i += blockDim.x) {
    float4 v = xr[i];
    const float4 a = sum_splits(ws, splits, (size_t)Mpad * N, (size_t)m * N + 4 * i);
    v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
    xr[i] = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)N + eps);
  const float4* wr = reinterpret_cast<const float4*>(w);
  __half2* o2 = reinterpret_cast<__half2*>(xn + (size_t)m * N);
  for (int i = threadIdx.x; i < N / 4; i += blockDim.x) {
    const float4 v = xr[i], g = wr[i];   // this thread's own row entries, written above
    o2[2 * i] = __floats2half2_rn(v.x * inv * g.x, v.y * inv * g.y);
    o2[2 * i + 1] = __floats2half2_rn(v.z * inv * g.z, v.w * inv * g.w);
  }
}

// ---- host side -------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// 2-D f16 map over a row-major [rows, cols] matrix, box = [box_rows, 64 cols], 128-byte swizzle.
// Cached by (pointer, rows, cols, box_rows).
bool make_map(CUtensorMap* out, const void* ptr, int rows, int cols, int box_rows) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int>, CUtensorMap> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_tuple(ptr, rows, cols, box_rows);
  auto itc = cache.find(key);
  if (itc != cache.end()) { *out = itc->second; return true; }
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache[key] = *out;
  return true;
}

}  // namespace tc

bool tensor_map(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* ptr, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  static std::mutex mu;
  static std::map<std::vector<uint64_t>, CUtensorMap> cache;
  if (rank < 1 || rank > 5) return false;
  std::vector<uint64_t> key{(uint64_t)dtype, (uint64_t)rank, (uint64_t)(uintptr_t)ptr, (uint64_t)swizzle};
  for (int i = 0; i < rank; ++i) key.push_back(dims[i]);
  for (int i = 0; i + 1 < rank; ++i) key.push_back(strides[i]);
  for (int i = 0; i < rank; ++i) key.push_back(box[i]);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) { *out = it->second; return true; }
  tc::EncodeTiledFn enc = tc::get_encode();
  if (!enc) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; e[i] = 1; }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  CUresult r = enc(out, dtype, (cuuint32_t)rank, const_cast<void*>(ptr), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache[key] = *out;
  return true;
}

namespace tc {

struct Plan {
  int bn, m_tiles, n_tiles, splits, kb_per_split, kb_total, units, grid;
  int pair;   // 1: CTA-pair kernel (256-row tiles, cta_group::2); bn is the pair's tile width
};

inline int max_ctas_of(int bn, int num_sms);

// The single-CTA plan of a fixed tile width without a K split.
inline Plan plan_with(int M, int N, int K, int bn) {
  const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + bn - 1) / bn, kb = K / BK;
  return Plan{bn, m_tiles, n_tiles, 1, kb, kb, m_tiles * n_tiles, 0, 0};
}

// The CTA-pair plan of tile width bn (no K split): m_tiles counts 128-row halves, units pairs.
inline Plan plan_pair(int M, int N, int K, int bn) {
  const int m_pairs = (M + 2 * BM - 1) / (2 * BM), n_tiles = (N + bn - 1) / bn, kb = K / BK;
  return Plan{bn, 2 * m_pairs, n_tiles, 1, kb, kb, m_pairs * n_tiles, 0, 1};
}

inline int max_pairs_of(int bn, int num_sms);

// Heuristic choice among the pair plans: fewest waves of pairs x tile width.
inline Plan plan_pair_for(int M, int N, int K, int epi, int num_sms) {
  const int cands[5] = {256, 208, 192, 176, 128};
  Plan best{};
  double best_cost = 1e30;
  const char* fb = getenv("S1_GEMM_BN");   // measurement / test override of the tile width
  const int force_bn = fb ? atoi(fb) : -1;
  for (int bn : cands) {
    if (epi == EPI_SWIGLU && (bn % 32)) continue;   // SwiGLU tiles hold whole 32-row gate/up groups
    if (force_bn > 0 && bn != force_bn) continue;
    const Plan pl = plan_pair(M, N, K, bn);
    const int maxp = max_pairs_of(bn, num_sms);
    const int waves = (pl.units + maxp - 1) / maxp;
    const double cost = (double)waves * (bn + 32.0);
    if (cost < best_cost * 0.999) { best_cost = cost; best = pl; }
  }
  return best;
}

// Few rows (at most two m tiles: questions over a snapshot) stream the weights: the estimated
// time in microseconds of a plan is a fixed launch and ramp cost, then the longer of the weight
// bytes at HBM speed and one CTA's share of k blocks (about 0.32 us per 64-deep block of 128
// weight rows), plus the split-K reduction when K is split. Fitted to cold-cache launch times of
// the 4B and 27B decide shapes over tile widths 128..256 and splits 1..8; ties (within 3 %) go
// to the narrower tile and the smaller split.
static double few_rows_cost_us(int N, int K, int bn, int kbp, int sp, int units, int maxc) {
  const double hbm_us = (double)N * K * 2 / 6.7e6;
  const int rounds = (units + maxc - 1) / maxc;
  const double stream_us = (double)rounds * kbp * 0.32 * bn / 128.0;
  return 5.0 + (hbm_us > stream_us ? hbm_us : stream_us) + (sp > 1 ? 6.0 + sp : 0.0);
}

// Choose the N tile and the K split together: minimise (waves of work units) x (k blocks per
// unit) x (per-k-block cost of the tile); few-row shapes by few_rows_cost_us.
Plan plan_for(int M, int N, int K, int epi, int num_sms, size_t ws_cap) {
  Plan best{};
  double best_cost = 1e30;
  const int kb_total = K / BK;
  const int m_tiles = (M + BM - 1) / BM;
  const char* fb0 = getenv("S1_GEMM_BN");
  const char* fs0 = getenv("S1_GEMM_SPLITS");
  if (m_tiles <= 2 && !fb0 && !fs0) {
    for (int bn : {128, 144, 176, 192, 208, 256}) {
      if (epi == EPI_SWIGLU && (bn % 32)) continue;
      const int n_tiles = (N + bn - 1) / bn;
      const int maxc = max_ctas_of(bn, num_sms);
      for (int sp = 1; sp <= 4; ++sp) {
        if (sp > 1 && kb_total / sp < 4) break;
        const int kbp = (kb_total + sp - 1) / sp;
        if ((kb_total + kbp - 1) / kbp != sp) continue;
        if (sp > 1 && (size_t)sp * m_tiles * BM * (size_t)N > ws_cap) break;
        const int units = m_tiles * n_tiles * sp;
        const double cost = few_rows_cost_us(N, K, bn, kbp, sp, units, maxc);
        if (cost < best_cost * 0.97) {
          best_cost = cost;
          best = Plan{bn, m_tiles, n_tiles, sp, kbp, kb_total, units, 0, 0};
        }
      }
    }
    if (best.bn != 0) return best;
  }
  // (176 and 208 are autotuner candidates only: measured slower than 144 in the split-K,
  // few-row weight-streaming plans this heuristic chooses; S1_GEMM_BN may still pin them)
  const int cands[6] = {256, 192, 144, 128, 208, 176};
  const char* fb = getenv("S1_GEMM_BN");   // measurement / test override of the tile width
  const int force_bn = fb ? atoi(fb) : -1;
  const char* fs = getenv("S1_GEMM_SPLITS");   // measurement override of the K split
  const int force_sp = fs ? atoi(fs) : -1;
  for (int bn : cands) {
    if (epi == EPI_SWIGLU && (bn % 32)) continue;
    if (force_bn > 0 ? bn != force_bn : (bn == 208 || bn == 176)) continue;
    const int n_tiles = (N + bn - 1) / bn;
    const int maxc = max_ctas_of(bn, num_sms);
    for (int splits = 1; splits <= 16; ++splits) {
      if (splits > 1 && (kb_total / splits) < 4) break;
      const int kbp = (kb_total + splits - 1) / splits;
      const int sp = (kb_total + kbp - 1) / kbp;
      if (sp != splits) continue;
      if (sp > 1 && (size_t)sp * m_tiles * BM * (size_t)N > ws_cap) break;
      const int units = m_tiles * n_tiles * sp;
      const int waves = (units + maxc - 1) / maxc;
      double cost = (double)waves * kbp * (bn + 48.0);
      if (sp > 1) cost *= 1.0 + 0.04 * sp;
      if ((force_sp <= 0 || sp == force_sp) && cost < best_cost * 0.999) {
        best_cost = cost;
        best = Plan{bn, m_tiles, n_tiles, sp, kbp, kb_total, units, 0, 0};
      }
      if (force_sp <= 0 && units >= maxc) break;
    }
  }
  if (best.bn == 0) best = plan_with(M, N, K, 128);   // (an override no candidate satisfies)
  return best;
}

template <int BN>
cudaLaunchConfig_t launch_config(cudaLaunchAttribute* attr, cudaStream_t st, bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Cfg<BN>::SMEM;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

// CTAs of this tile width that fit on the GPU at once (queried once, then cached).
template <int BN>
int max_ctas(int num_sms) {
  static int cached = -1;
  if (cached < 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN>::SMEM);
    int per_sm = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_kernel<BN>, NUM_THREADS, Cfg<BN>::SMEM);
    if (e != cudaSuccess || per_sm <= 0) {
      cudaGetLastError();
      per_sm = 1;
    }
    cached = per_sm * num_sms;
  }
  return cached;
}

inline int max_ctas_of(int bn, int num_sms) {
  switch (bn) {
    case 256: return max_ctas<256>(num_sms);
    case 208: return max_ctas<208>(num_sms);
    case 192: return max_ctas<192>(num_sms);
    case 176: return max_ctas<176>(num_sms);
    case 144: return max_ctas<144>(num_sms);
    default: return max_ctas<128>(num_sms);
  }
}

template <int BN>
cudaLaunchConfig_t launch_config_pair(cudaLaunchAttribute* attr, cudaStream_t st, bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Cfg2<BN>::SMEM;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

// CTA pairs of this tile width that fit on the GPU at once (queried once, then cached).
template <int BN>
int max_pairs(int num_sms) {
  static int cached = -1;
  if (cached < 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg2<BN>::SMEM);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config_pair<BN>(attr, 0);
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int n = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<BN>, &cfg);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    cached = n;
  }
  return cached;
}

inline int max_pairs_of(int bn, int num_sms) {
  switch (bn) {
    case 256: return max_pairs<256>(num_sms);
    case 208: return max_pairs<208>(num_sms);
    case 192: return max_pairs<192>(num_sms);
    case 176: return max_pairs<176>(num_sms);
    default: return max_pairs<128>(num_sms);
  }
}

template <int BN>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, Params p, int num_sms,
                        cudaStream_t st) {
  const int mp = max_pairs<BN>(num_sms);
  cudaLaunchAttribute attr[2];
  const bool pdl = pdl_enabled();
  cudaLaunchConfig_t cfg = launch_config_pair<BN>(attr, st, pdl);
  p.m_groups = p.m_tiles / 2;
  p.units = p.m_groups * p.splits * p.n_tiles;
  const int ncl = p.units < mp ? p.units : mp;
  cfg.gridDim = dim3(2 * ncl);
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<BN>, ma, mb, mo, p);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, Params p, int num_sms,
                      cudaStream_t st) {
  const int mc = max_ctas<BN>(num_sms);
  cudaLaunchAttribute attr[1];
  const bool pdl = pdl_enabled();
  cudaLaunchConfig_t cfg = launch_config<BN>(attr, st, pdl);
  p.m_groups = p.m_tiles;
  p.units = p.m_groups * p.splits * p.n_tiles;
  cfg.gridDim = dim3(p.units < mc ? p.units : mc);
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN>, ma, mb, mo, p);
}

}  // namespace tc

bool gemm_tc_supported(int M, int N, int K, int epi) {
  return M >= 0 && N > 0 && K > 0 && (K % tc::BK) == 0 && (N % 32) == 0 && epi >= 0 && epi <= 3 &&
         tc::get_encode() != nullptr;
}

size_t gemm_tc_plan_ws_floats(int M, int N, int K, int epi, int num_sms, size_t ws_cap) {
  const tc::Plan pl = tc::plan_for(M, N, K, epi, num_sms, ws_cap);
  return pl.splits > 1 ? (size_t)pl.splits * pl.m_tiles * tc::BM * (size_t)N : 0;
}

size_t gemm_tc_workspace_floats(int M, int N, int K, int epi, int num_sms) {
  // K is split only while the tile count is below the SM count, so the partials of one
  // launch never exceed about 2 x num_sms tiles of 128 x 256.
  (void)M; (void)N; (void)K; (void)epi;
  return (size_t)2 * (num_sms > 0 ? num_sms : 160) * tc::BM * 256;
}

static cudaError_t launch_plan(const tc::Plan& pl, const f16* X, const f16* W, int M, int N, int K, int epi,
                               void* out, int ldo, float* splitk_ws, const LaunchCtx& lc) {
  CUtensorMap ma, mb;
  const int brows = pl.pair ? pl.bn / 2 : pl.bn;
  if (!tc::make_map(&ma, X, M, K, tc::BM) || !tc::make_map(&mb, W, N, K, brows)) return cudaErrorInvalidValue;
  tc::Params p;
  p.M = M; p.N = N; p.K = K;
  p.m_tiles = pl.m_tiles; p.n_tiles = pl.n_tiles; p.splits = pl.splits;
  p.kb_per_split = pl.kb_per_split; p.kb_total = pl.kb_total;
  p.m_groups = 0; p.units = 0;   // set by the launcher for its kernel family
  p.epi = pl.splits > 1 ? tc::EPI_PARTIAL : epi;
  p.out = out; p.ldo = ldo; p.ws = splitk_ws; p.d_err = lc.d_err;
  // fp32 output map: 32-row x 16-column boxes (64-byte rows, 64-byte swizzle), matching the
  // epilogue's staging layout
  CUtensorMap mo;
  {
    const bool part = pl.splits > 1;
    if (part || epi == EPI_F32 || epi == EPI_RESADD) {
      const uint64_t rows = part ? (uint64_t)pl.splits * pl.m_tiles * tc::BM : (uint64_t)M;
      const uint64_t pitch = part ? (uint64_t)N * 4 : (uint64_t)ldo * 4;
      const void* base = part ? (const void*)p.ws : out;
      if ((pitch % 16) != 0 || ((uintptr_t)base % 16) != 0) return cudaErrorInvalidValue;
      const uint64_t dims[2] = {(uint64_t)N, rows};
      const uint64_t strides[1] = {pitch};
      const uint32_t box[2] = {16, 32};
      if (!tensor_map(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    } else {
      memset(&mo, 0, sizeof(mo));   // f16 outputs are stored from registers
    }
  }
  cudaError_t e;
  if (pl.pair) {
    switch (pl.bn) {
      case 256: e = tc::launch_pair<256>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
      case 208: e = tc::launch_pair<208>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
      case 192: e = tc::launch_pair<192>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
      case 176: e = tc::launch_pair<176>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
      default: e = tc::launch_pair<128>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
    }
  } else switch (pl.bn) {
    case 256: e = tc::launch_bn<256>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
    case 208: e = tc::launch_bn<208>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
    case 192: e = tc::launch_bn<192>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
    case 176: e = tc::launch_bn<176>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
    case 144: e = tc::launch_bn<144>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
    default: e = tc::launch_bn<128>(ma, mb, mo, p, lc.num_sms, lc.stream); break;
  }
  if (lc.launches) *lc.launches += 1;
  if (e != cudaSuccess || pl.splits == 1) return e;
  if (epi == EPI_RESADD && lc.norm_w && lc.norm_out && M <= 512 && N % 4 == 0) {
    CK_RET(launch_pdl(tc::splitk_resadd_norm_kernel, dim3(M), dim3(norm_row_threads(N)), 0, lc.stream, p.ws, pl.splits,
                      pl.m_tiles * tc::BM, N, (float*)out, ldo, lc.norm_w, lc.norm_out, lc.norm_eps));
    if (lc.launches) *lc.launches += 1;
    if (lc.norm_done) *lc.norm_done = true;
    return cudaGetLastError();
  }
  const int cols = epi == EPI_SWIGLU ? N / 2 : N;
  const size_t work = (size_t)M * cols / 4;
  int blocks = (int)((work + 255) / 256);
  if (blocks > 4 * lc.num_sms) blocks = 4 * lc.num_sms;
  CK_RET(launch_pdl(tc::splitk_reduce_kernel, dim3(blocks), dim3(256), 0, lc.stream, p.ws, pl.splits,
                    pl.m_tiles * tc::BM, M, N, epi, out, ldo));
  if (lc.launches) *lc.launches += 1;
  return cudaGetLastError();
}

namespace tc {
// Measured choice of (BN, pair) per GEMM shape for plans without a K split. Every such plan
// accumulates each output over K in the same order, so the choice never changes results.
struct Tuned { int bn, pair; };
std::mutex g_tune_mu;
std::map<std::tuple<int, int, int, int, int, int>, Tuned> g_tuned;

bool tune_enabled() {
  const char* e = getenv("S1_GEMM_TUNE");
  return !(e && e[0] == '0');
}

// Which kernel families a launch may use: the caller's variant, narrowed by the S1_GEMM_PAIR
// measurement override ("0": single-CTA only, "1": CTA pairs only).
int variant_of(const LaunchCtx& lc) {
  if (lc.variant != GEMM_ANY) return lc.variant;
  const char* e = getenv("S1_GEMM_PAIR");
  if (e && e[0] == '0') return GEMM_SINGLE;
  if (e && e[0] == '1') return GEMM_PAIR;
  return GEMM_ANY;
}

inline Plan plan_of(int M, int N, int K, const Tuned& t) {
  return t.pair ? plan_pair(M, N, K, t.bn) : plan_with(M, N, K, t.bn);
}

// Times every candidate (single-CTA BN, and CTA-pair BN) three times on the caller's stream
// from a flushed L2 (tuning output `scratch`, RESADD shapes tuned with a plain fp32 store of the
// same size) and keeps the fastest of the last two runs.
cudaError_t tune(Plan& pl, const f16* X, const f16* W, int M, int N, int K, int epi, void* out, int ldo,
                 const LaunchCtx& lc, int variant) {
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, M, N, K, epi, variant);
  {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    auto it = g_tuned.find(key);
    if (it != g_tuned.end()) {
      pl = plan_of(M, N, K, it->second);
      return cudaSuccess;
    }
  }
  const bool resadd = epi == EPI_RESADD;
  void* tout = resadd ? lc.tune_out : out;
  const int tldo = resadd ? N : ldo;
  const int tepi = resadd ? EPI_F32 : epi;
  if (!tout || (resadd && (size_t)M * N > lc.tune_floats)) return cudaSuccess;   // keep the heuristic plan
  LaunchCtx l2 = lc;
  l2.launches = nullptr;
  // Each timed run starts with L2 flushed (the caller's buffer, larger than L2, rewritten), as in
  // a forward pass, where every weight tile comes from DRAM. Without a buffer the runs are timed
  // from a warm L2.
  void* flush = lc.tune_flush;
  const size_t flush_bytes = lc.tune_flush_bytes;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return cudaGetLastError();
  if (cudaEventCreate(&e1) != cudaSuccess) { cudaEventDestroy(e0); return cudaGetLastError(); }
  float best = 1e30f;
  Tuned bt{pl.bn, pl.pair};
  std::vector<Tuned> cands;
  if (variant != GEMM_PAIR)
    for (int bn : {256, 208, 192, 176, 144, 128})
      if (!(epi == EPI_SWIGLU && (bn % 32))) cands.push_back(Tuned{bn, 0});
  // (CTA pairs only when there are more rows than one single-CTA tile: with at most 128 rows a
  // pair's 256-row tile is more than half padding)
  if (variant != GEMM_SINGLE && (M > BM || variant == GEMM_PAIR))
    for (int bn : {256, 208, 192, 176, 128})
      if (!(epi == EPI_SWIGLU && (bn % 32))) cands.push_back(Tuned{bn, 1});
  cudaError_t err = cudaSuccess;
  for (const Tuned& c : cands) {
    if (err != cudaSuccess) break;
    const Plan cand = plan_of(M, N, K, c);
    float t = 1e30f;
    for (int rep = 0; rep < 3 && err == cudaSuccess; ++rep) {
      if (flush) cudaMemsetAsync(flush, rep, flush_bytes, lc.stream);
      cudaEventRecord(e0, lc.stream);
      err = launch_plan(cand, X, W, M, N, K, tepi, tout, tldo, nullptr, l2);
      cudaEventRecord(e1, lc.stream);
      if (err == cudaSuccess) err = cudaEventSynchronize(e1);
      float ms = 0.f;
      if (err == cudaSuccess && rep > 0 && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess) t = std::min(t, ms);
    }
    if (getenv("S1_GEMM_TUNE_LOG") && getenv("S1_GEMM_TUNE_LOG")[0] == '2')
      fprintf(stderr, "gemm cand M=%d N=%d K=%d epi=%d %s bn=%d %.2f us\n", M, N, K, epi,
              c.pair ? "pair" : "single", c.bn, 1e3f * t);
    if (t < best) { best = t; bt = c; }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tuned[key] = bt;
  }
  if (getenv("S1_GEMM_TUNE_LOG"))
    fprintf(stderr, "gemm tune M=%d N=%d K=%d epi=%d -> %s bn=%d (%.2f us)\n", M, N, K, epi,
            bt.pair ? "pair" : "single", bt.bn, 1e3f * best);
  pl = plan_of(M, N, K, bt);
  return cudaSuccess;
}
}  // namespace tc

cudaError_t launch_gemm_tc(const f16* X, const f16* W, int M, int N, int K, int epi, void* out, int ldo,
                           float* splitk_ws, size_t ws_floats, const LaunchCtx& lc) {
  if (M == 0) return cudaSuccess;
  if (!gemm_tc_supported(M, N, K, epi)) return cudaErrorInvalidValue;
  const int variant = tc::variant_of(lc);
  tc::Plan pl = variant == GEMM_PAIR ? tc::plan_pair_for(M, N, K, epi, lc.num_sms)
                                     : tc::plan_for(M, N, K, epi, lc.num_sms, splitk_ws ? ws_floats : 0);
  // (at most 128 rows: the planner's streaming model was fitted to measured launches of these
  // shapes, and the tuner's short timings would only add noise)
  if (pl.splits == 1 && lc.tune && tc::tune_enabled() && !getenv("S1_GEMM_BN") && M > tc::BM) {
    cudaError_t e = tc::tune(pl, X, W, M, N, K, epi, out, ldo, lc, variant);
    if (e != cudaSuccess) return e;
  }
  return launch_plan(pl, X, W, M, N, K, epi, out, ldo, splitk_ws, lc);
}

cudaError_t launch_gemm_lse(const f16* X, const f16* W, int M, int N, int K, float2* part, int ldp,
                            const LaunchCtx& lc) {
  if (M <= 0) return cudaSuccess;
  if (!gemm_tc_supported(M, N, K, EPI_F32) || M > ldp || !part) return cudaErrorInvalidValue;
  const tc::Plan pl = tc::plan_with(M, N, K, GEMM_LSE_BN);
  return launch_plan(pl, X, W, M, N, K, EPI_LSE, part, ldp, nullptr, lc);
}

}  // namespace s1

// =======================================================================================
// GEMM entry point that allocates nothing.
//
// For callers that cannot allocate device memory at call time: code running where
// cudaMalloc is not allowed or not wanted (inside a real-time serving loop that must not
// synchronise the device, under an allocator that is owned by another framework, or in a
// process whose memory budget is fixed up front). Its split-K partials and its error word live
// in file-scope device arrays of a fixed size, reserved when the library is loaded; every
// GPU that loads the library holds them until the process exits.
#include "../../include/s1.h"
#include "../../include/s1_ops.h"

namespace s1 {
int set_error(int code, const char* msg);
}

namespace {
static __device__ __align__(256) float g_noalloc_ws[S1_NOALLOC_WS_FLOATS];
static __device__ __align__(256) int g_noalloc_err[64];

struct NoAllocDev {
  bool ready = false;
  float* ws = nullptr;   // device address of g_noalloc_ws on this device
  int* err = nullptr;    // device address of g_noalloc_err on this device
  int sms = 0;
};
std::mutex g_noalloc_mu;
NoAllocDev g_noalloc_dev[64];

// Set-up, once per device, with that device current: host code only has a stand-in for the
// arrays' names, so their device addresses are looked up here.
int noalloc_setup(int dev, NoAllocDev** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (dev < 0 || dev >= 64) return s1::set_error(S1_ERR_UNSUPPORTED, "gemm_noalloc: device index out of range");
  NoAllocDev& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess) return s1::set_error(S1_ERR_CUDA, "gemm_noalloc: cudaGetSymbolAddress(workspace) failed");
    d.ws = (float*)p;
    e = cudaGetSymbolAddress(&p, g_noalloc_err);
    if (e != cudaSuccess) return s1::set_error(S1_ERR_CUDA, "gemm_noalloc: cudaGetSymbolAddress(error word) failed");
    d.err = (int*)p;
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return s1::set_error(S1_ERR_CUDA, "gemm_noalloc: device query failed");
    d.ready = true;
  }
  *out = &d;
  return S1_OK;
}
}  // namespace

extern "C" int s1_op_gemm_noalloc(const void* X, const void* W, int32_t M, int32_t N, int32_t K, int32_t epi,
                                  void* out, int32_t ldo, void* stream) {
  using namespace s1;
  cudaStream_t st = (cudaStream_t)stream;
  if (M < 0 || N <= 0 || K <= 0 || K % 64 || N % 32 || epi < 0 || epi > 3 || !X || !W || !out)
    return set_error(S1_ERR_INVALID_ARG, "gemm_noalloc: bad sizes, epilogue or NULL pointer");
  if (!gemm_tc_supported(M, N, K, epi)) return set_error(S1_ERR_UNSUPPORTED, "gemm_noalloc: shape not supported");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_error(S1_ERR_CUDA, "gemm_noalloc: no current device");
  NoAllocDev* d = nullptr;
  int rc = noalloc_setup(dev, &d);
  if (rc) return rc;
  // Same plan as s1_op_gemm (so the two give identical results); its split-K partials must
  // fit the fixed array.
  const size_t plan_cap = gemm_tc_workspace_floats(M, N, K, epi, d->sms);
  const size_t need = gemm_tc_plan_ws_floats(M, N, K, epi, d->sms, plan_cap);
  if (need > (size_t)S1_NOALLOC_WS_FLOATS) {
    char msg[200];
    snprintf(msg, sizeof(msg), "gemm_noalloc: this shape needs %zu floats of split-K scratch, more than the %d reserved",
             need, (int)S1_NOALLOC_WS_FLOATS);
    return set_error(S1_ERR_BUDGET, msg);
  }
  if (cudaMemsetAsync(d->err, 0, sizeof(int), st) != cudaSuccess)
    return set_error(S1_ERR_CUDA, "gemm_noalloc: clearing the error word failed");
  LaunchCtx lc{st, d->err, d->sms, nullptr};
  // the plan writes only `need` floats of the array; plan_cap only selects the same plan
  cudaError_t e = launch_gemm_tc((const f16*)X, (const f16*)W, M, N, K, epi, out, ldo, d->ws, plan_cap, lc);
  if (e != cudaSuccess) return set_error(S1_ERR_CUDA, cudaGetErrorString(e));
  int h = 0;
  if (cudaMemcpyAsync(&h, d->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return set_error(S1_ERR_CUDA, "gemm_noalloc: synchronisation failed");
  if (h) return set_error(S1_ERR_DEVICE_TIMEOUT, "gemm_noalloc: a bounded device wait gave up");
  return S1_OK;
}

extern "C" int s1_gemm_plan(int32_t M, int32_t N, int32_t K, int32_t epi, int32_t num_sms, int32_t pair,
                            int32_t* out) {
  using namespace s1;
  if (!out || M < 1 || N < 32 || N % 32 || K < 64 || K % 64 || epi < 0 || epi > 3 || num_sms < 1)
    return set_error(S1_ERR_INVALID_ARG, "gemm_plan: bad sizes, epilogue, SM count or NULL output");
  const tc::Plan pl = pair ? tc::plan_pair_for(M, N, K, epi, num_sms)
                           : tc::plan_for(M, N, K, epi, num_sms, gemm_tc_workspace_floats(M, N, K, epi, num_sms));
  out[0] = pl.bn;
  out[1] = 1;   // CTAs per weight tile (no clusters along M)
  out[2] = pl.pair;
  out[3] = pl.splits;
  out[4] = pl.kb_per_split;
  out[5] = pl.m_tiles;
  out[6] = pl.n_tiles;
  return S1_OK;
}
