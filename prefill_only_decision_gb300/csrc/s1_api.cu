// libs1: executor and C ABI.
//
// The executor owns the device weights (LoRA merged at load, packed for the fused
// projections), the per-call scratch, and the launch sequence of one forward pass over
// packed rows on one stream. A state (prefix snapshot) owns the per-layer gated
// delta-rule states (fp32) and full-attention K/V (f16, post-RoPE).
#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "common.cuh"
#include "../../include/s1.h"
#include "../../include/s1_ops.h"

using namespace s1;

// ---------------------------------------------------------------------------------------
// errors and allocation
namespace {
thread_local std::string g_err;
// Device allocator: the hooks installed by s1_set_allocator (NULL: cudaMalloc / cudaFree). A model
// keeps the hooks that were installed when it was created, and every allocation and free made on
// its behalf goes through them (t_alloc points at them for the duration of each call on it), so
// installing other hooks later never frees its blocks through the wrong allocator.
struct Alloc {
  void* (*alloc)(size_t, void*) = nullptr;
  void (*free)(void*, void*) = nullptr;
  void* ctx = nullptr;
};
Alloc g_al;
thread_local const Alloc* t_alloc = nullptr;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

void* dalloc(size_t bytes) {
  if (bytes == 0) bytes = 256;
  const Alloc& a = t_alloc ? *t_alloc : g_al;
  if (a.alloc) return a.alloc(bytes, a.ctx);
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}
void dfree(void* p) {
  if (!p) return;
  const Alloc& a = t_alloc ? *t_alloc : g_al;
  if (a.free) a.free(p, a.ctx);
  else cudaFree(p);
}

#define CK(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) return fail(S1_ERR_CUDA, "%s: %s (%s:%d)", #call,              \
                                       cudaGetErrorString(e_), __FILE__, __LINE__);       \
  } while (0)

constexpr uint32_t MODEL_MAGIC = 0x5331304du, STATE_MAGIC = 0x53315354u, DEAD = 0xdeadbeefu;
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

namespace s1 {
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace s1

// ---------------------------------------------------------------------------------------
struct Layer {
  bool full;
  int ord;             // index among layers of its kind
  float* attn_norm;
  float* mlp_norm;
  f16 * w_in;          // packed in-projection
  int n_in;
  f16 * w_o;
  int k_o;             // in-features of w_o
  f16 * w_gu;          // [2F, d], gate/up interleaved by 16 rows
  f16 * w_down;        // [d, F]
  float* conv_w;       // gated delta rule's short convolution taps [2*H*dk + H*dv, width] (or NULL)
};

struct Scratch {
  int rows = 0;
  int opt_cap = 0;           // option ids the metadata / output blocks hold
  float* x = nullptr;
  f16 * xn = nullptr;
  float* proj = nullptr;
  f16 * mix = nullptr;
  f16 * h = nullptr;
  f16 * q = nullptr;
  f16 * knew = nullptr;
  f16 * vnew = nullptr;
  float* loga = nullptr;
  float* beta = nullptr;
  void* gdn = nullptr;       // chunked scan, per row: normalised k, W, Ut, K' (f16 [R, H, dk] each)
  float* projc = nullptr;    // gated delta rule's in-projection after the short convolution (or NULL)
  int* meta = nullptr;       // row_src | row_seq | seqs | ctxs | readout metadata
  size_t meta_bytes = 0;
  float* ws = nullptr;       // split-K workspace
  size_t ws_floats = 0;
  float* out = nullptr;      // readout outputs for the blocking API
  size_t out_floats = 0;
  std::vector<void*> blocks;
};

struct s1_model {
  uint32_t magic;
  Alloc al;   // the allocator hooks of this model's device memory (those installed at creation)
  s1_shape sh;
  std::vector<uint8_t> is_full;
  int nG = 0, nF = 0, n_in_gdn = 0, n_in_fa = 0, n_proj = 0, n_mix = 0;
  int device = 0, num_sms = 0;
  cudaStream_t stream = nullptr;
  void* arena = nullptr;
  f16* embed = nullptr;          // tied embedding, f16 copy
  float* final_norm = nullptr;
  std::vector<Layer> layers;
  float2* rope_tab = nullptr;
  int max_pos = 0;
  int* d_err = nullptr;
  Scratch sc;
  float* lm_buf = nullptr;     // full-vocabulary option log-probabilities: lm | z | h_hat | partials
  size_t lm_floats = 0;
  void* schunk = nullptr;      // chunked scan, per chunk: B, N^T and the start state ([chunks, H, dk, dk])
  size_t schunk_chunks = 0;
  void* tune_flush = nullptr;  // GEMM autotuner: L2-flush buffer (allocated with the model)
  size_t tune_flush_bytes = 0;
  bool gdn_token = false;      // S1_GDN=token: token-by-token scan (debugging)
  bool attn_sync = false;      // S1_ATTN=sync: mma.sync attention kernel (debugging)
  char* pinned = nullptr;      // host staging for metadata uploads
  size_t pinned_bytes = 0;
  cudaEvent_t meta_done = nullptr;
  int gemm_impl = 0;           // 0 = tensor cores (tcgen05), 1 = SIMT reference
  float* trace = nullptr;      // layer trace: residual stream after the embedding and each layer
  long long trace_floats = 0;
  bool force_simt = false;     // S1_GEMM=simt in the environment (debugging)
  bool vocab_simt = false;     // S1_VOCAB=simt: full-vocabulary pass on CUDA cores
  bool fuse_norm = true;       // RMSNorm fused into split-K residual reductions (S1_NORM_FUSE=0: off)
  // profiling
  bool prof = false;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> prof_ev;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_next = 0;
  double prof_flops[S1_PROF_NCLASS] = {0};
  double prof_bytes[S1_PROF_NCLASS] = {0};
  long prof_count[S1_PROF_NCLASS] = {0};
  long launches = 0;           // kernels launched by forward passes
  long long h2d_bytes = 0, d2h_bytes = 0;
  // CUDA graphs of the stream-ordered calls (s1_set_graphs): keyed by the call's argument
  // signature; a graph owns its metadata buffer and bakes in the scratch addresses. Both sets
  // are bounded (kMaxGraphs captured graphs; the seen-once set is cleared at kMaxSeen entries),
  // so callers whose signatures never repeat cost no memory growth.
  struct Graph {
    cudaGraphExec_t exec = nullptr;
    void* meta = nullptr;
    long launches = 0;
  };
  static constexpr size_t kMaxGraphs = 64, kMaxSeen = 4096;
  bool graphs = false;
  std::map<std::string, Graph> graph_cache;
  std::set<std::string> graph_seen;
};

// Every captured graph is dropped when a buffer it uses moves (scratch or chunk-state growth)
// or when graphs are switched off.
void drop_graphs(s1_model* m) {
  for (auto& kv : m->graph_cache) {
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    dfree(kv.second.meta);
  }
  m->graph_cache.clear();
  m->graph_seen.clear();
}

struct s1_state {
  uint32_t magic;
  s1_model* model;
  int P, cap;
  float* S;
  f16 * KV;
  float* conv;         // short-convolution history [n_gdn_layers, width - 1, channels] (or NULL)
  void* mem;
  Alloc al;            // the hooks `mem` came from (its model's)
};

// ---------------------------------------------------------------------------------------
// profiling helpers
namespace {
cudaEvent_t next_event(s1_model* m) {
  if (m->ev_next == m->ev_pool.size()) {
    cudaEvent_t e;
    cudaEventCreate(&e);
    m->ev_pool.push_back(e);
  }
  return m->ev_pool[m->ev_next++];
}
struct ProfScope {
  s1_model* m;
  int cls;
  cudaEvent_t b = nullptr;
  ProfScope(s1_model* m_, int cls_, double flops, double bytes) : m(m_), cls(cls_) {
    if (!m->prof) return;
    b = next_event(m);
    cudaEventRecord(b, m->stream);
    m->prof_flops[cls] += flops;
    m->prof_bytes[cls] += bytes;
    m->prof_count[cls] += 1;
  }
  ~ProfScope() {
    if (!m->prof) return;
    cudaEvent_t e = next_event(m);
    cudaEventRecord(e, m->stream);
    m->prof_ev.push_back({cls, {b, e}});
  }
};
}  // namespace

// ---------------------------------------------------------------------------------------
// scratch management
namespace {
size_t meta_bytes_for(int rows, int max_seq, int max_ctx, int max_q, int max_opt) {
  return align_up((size_t)rows * 2 * sizeof(int), 256) + align_up((size_t)max_seq * sizeof(SeqDesc), 256) +
         align_up((size_t)(rows + max_seq) * sizeof(ChunkDesc), 256) +
         align_up((size_t)max_ctx * sizeof(CtxDesc), 256) + align_up((size_t)max_ctx * attention_ctx_map_bytes(), 256) +
         align_up((size_t)(3 * max_q + 1 + max_opt) * sizeof(int), 256);
}

void free_scratch(Scratch& sc) {
  for (void* p : sc.blocks) dfree(p);
  sc = Scratch();
}

int ensure_scratch(s1_model* m, int rows, int n_opts = 0) {
  if (rows <= m->sc.rows && n_opts <= m->sc.opt_cap) return S1_OK;
  rows = std::max(rows, m->sc.rows);
  int want = std::max(rows, 256);
  want = std::min(std::max(want, m->sc.rows * 2), m->sh.max_rows);
  want = std::max(want, rows);
  CK(cudaStreamSynchronize(m->stream));
  drop_graphs(m);
  free_scratch(m->sc);
  Scratch sc;
  const s1_shape& s = m->sh;
  auto take = [&](size_t bytes) -> void* {
    void* p = dalloc(align_up(bytes, 1024));
    if (p) sc.blocks.push_back(p);
    return p;
  };
  const size_t R = (size_t)want;
  const int H = s.la_heads > 0 ? s.la_heads : 1;
  sc.x = (float*)take(R * s.d_model * 4);
  sc.xn = (f16*)take(R * s.d_model * 2);
  sc.proj = (float*)take(R * m->n_proj * 4);
  sc.mix = (f16*)take(R * m->n_mix * 2);
  sc.h = (f16*)take(R * s.ffn * 2);
  sc.q = (f16*)take(R * (size_t)s.fa_q_heads * s.fa_head_dim * 2 + 256);
  sc.knew = (f16*)take(R * (size_t)s.fa_kv_heads * s.fa_head_dim * 2 + 256);
  sc.vnew = (f16*)take(R * (size_t)s.fa_kv_heads * s.fa_head_dim * 2 + 256);
  sc.loga = (float*)take(R * H * 4);
  sc.beta = (float*)take(R * H * 4);
  sc.gdn = take(R * gdn_row_bytes(H, std::max(s.la_dk, 1)));
  if (s.conv_width > 0 && m->n_in_gdn > 0) {
    sc.projc = (float*)take(R * m->n_in_gdn * 4);
    if (!sc.projc) {
      free_scratch(sc);
      return fail(S1_ERR_OOM, "scratch allocation for %d rows failed", want);
    }
  }
  const int max_seq = want, max_ctx = want, max_q = want;
  const int max_opt = std::max(64 * want, std::max(n_opts, m->sc.opt_cap));
  sc.opt_cap = max_opt;
  sc.meta_bytes = meta_bytes_for(want, max_seq, max_ctx, max_q, max_opt);
  sc.meta = (int*)take(sc.meta_bytes);
  sc.ws_floats = std::max<size_t>(gemm_tc_workspace_floats(want, std::max(m->n_proj, 2 * s.ffn), s.ffn, EPI_RESADD, m->num_sms), 1);
  sc.ws = (float*)take(sc.ws_floats * 4);
  sc.out_floats = (size_t)max_opt + (size_t)max_q * S1_STAT_COUNT + (size_t)max_q * s.d_model;
  sc.out = (float*)take(sc.out_floats * 4);
  for (void* p : {(void*)sc.x, (void*)sc.xn, (void*)sc.proj, (void*)sc.mix, (void*)sc.h, (void*)sc.q,
                  (void*)sc.knew, (void*)sc.vnew, (void*)sc.loga, (void*)sc.beta, sc.gdn,
                  (void*)sc.meta,
                  (void*)sc.ws, (void*)sc.out}) {
    if (!p) {
      free_scratch(sc);
      return fail(S1_ERR_OOM, "scratch allocation for %d rows failed", want);
    }
  }
  sc.rows = want;
  m->sc = sc;
  if (m->pinned_bytes < sc.meta_bytes) {
    if (m->pinned) cudaFreeHost(m->pinned);
    m->pinned = nullptr;
    if (cudaMallocHost((void**)&m->pinned, sc.meta_bytes) != cudaSuccess) {
      cudaGetLastError();
      m->pinned_bytes = 0;
      return fail(S1_ERR_OOM, "pinned staging allocation failed");
    }
    m->pinned_bytes = sc.meta_bytes;
  }
  return S1_OK;
}

// Metadata of one forward call, assembled on the host and uploaded in one copy.
struct Meta {
  std::vector<int> row_src, row_seq;
  std::vector<SeqDesc> seqs;
  std::vector<CtxDesc> ctxs;
  std::vector<ChunkDesc> chunks;
  std::vector<int> q_row, q_type, opt_off, opt_ids;
  int max_len = 0, max_opts = 0;
  int n_first = 0;   // fused sweep: the first n_first sequences (prefixes) scan before the rest
  // sequences from fold_from on are handled by their prefixes' state pass, sequences from
  // out_fold on by the output kernel alone (see build_chunks)
  int fold_from = 0;
  int out_fold = 0;
  // device views
  int* d_row_src = nullptr;
  int* d_row_seq = nullptr;
  SeqDesc* d_seqs = nullptr;
  CtxDesc* d_ctxs = nullptr;
  void* d_ctx_maps = nullptr;   // attention's tensor map of each context's K/V (tcgen05 path)
  ChunkDesc* d_chunks = nullptr;
  int *d_q_row = nullptr, *d_q_type = nullptr, *d_opt_off = nullptr, *d_opt_ids = nullptr;
};

// Splits every sequence into 64-row chunks (chunk boundaries restart at each sequence).
void build_chunks(Meta& mt) {
  mt.chunks.clear();
  for (size_t s = 0; s < mt.seqs.size(); ++s) {
    SeqDesc& sd = mt.seqs[s];
    sd.chunk0 = (int)mt.chunks.size();
    for (int c = 0; c < sd.len; c += GDN_CHUNK)
      mt.chunks.push_back(ChunkDesc{sd.row0 + c, std::min(GDN_CHUNK, sd.len - c), (int)s});
  }
  // Fused sweep: when every later sequence is a single chunk that keeps no state and continues
  // a prefix of this call (contiguously per prefix), the prefixes' state pass also records the
  // later sequences' start states, and they get no state pass of their own.
  const int n = (int)mt.seqs.size();
  mt.fold_from = n;
  mt.out_fold = n;
  if (mt.n_first <= 0 || mt.n_first >= n) {
    // one group (e.g. questions over snapshots): if every sequence is a single chunk that keeps
    // no state, the output kernel reads each chunk's start state from its snapshot and no state
    // pass runs
    bool all = true;
    for (int s = 0; s < n && all; ++s)
      if (mt.seqs[s].len > GDN_CHUNK || mt.seqs[s].ctx_out >= 0) all = false;
    if (all) mt.out_fold = 0;
  }
  if (mt.n_first > 0 && mt.n_first < n) {
    std::vector<int> owner(mt.ctxs.size(), -1);
    for (int p = 0; p < mt.n_first; ++p)
      if (mt.seqs[p].ctx_out >= 0 && mt.seqs[p].ctx_out < (int)owner.size()) owner[mt.seqs[p].ctx_out] = p;
    bool ok = true;
    for (int s = mt.n_first; s < n && ok; ++s) {
      const SeqDesc& q = mt.seqs[s];
      const int p = (q.ctx_in >= 0 && q.ctx_in < (int)owner.size()) ? owner[q.ctx_in] : -1;
      if (q.len > GDN_CHUNK || q.ctx_out >= 0 || p < 0) { ok = false; break; }
      SeqDesc& ps = mt.seqs[p];
      if (ps.fol1 <= ps.fol0) { ps.fol0 = s; ps.fol1 = s + 1; }
      else if (ps.fol1 == s) ps.fol1 = s + 1;
      else ok = false;
    }
    if (ok) {
      mt.fold_from = mt.n_first;
    } else {
      for (int p = 0; p < mt.n_first; ++p) mt.seqs[p].fol0 = mt.seqs[p].fol1 = 0;
    }
  }
}

// Packs the call's metadata and uploads it: through the pinned staging buffer into the scratch
// (stream-ordered), or, for a graph being captured, synchronously into the graph's own buffer
// `dest` of `dest_bytes` (allocated here when NULL; returned through `dest`).
int upload_meta(s1_model* m, Meta& mt, void** dest = nullptr) {
  build_chunks(mt);
  const int R = (int)mt.row_src.size();
  const size_t need = meta_bytes_for(R, (int)mt.seqs.size(), (int)mt.ctxs.size(), (int)mt.q_row.size(),
                                     (int)mt.opt_ids.size());
  if (need > m->sc.meta_bytes) return fail(S1_ERR_BUDGET, "request metadata exceeds the scratch budget");
  std::vector<char> stage;
  char* h;
  char* d;
  if (dest) {
    *dest = dalloc(need);
    if (!*dest) return fail(S1_ERR_OOM, "graph metadata allocation failed");
    stage.resize(need);
    h = stage.data();
    d = (char*)*dest;
  } else {
    // the previous upload from the pinned buffer must have finished before it is rewritten
    CK(cudaEventSynchronize(m->meta_done));
    h = m->pinned;
    d = (char*)m->sc.meta;
  }
  size_t off = 0;
  auto put = [&](const void* src, size_t bytes) -> char* {
    if (bytes) memcpy(h + off, src, bytes);
    char* dp = d + off;
    off += align_up(bytes, 256);
    return dp;
  };
  mt.d_row_src = (int*)put(mt.row_src.data(), R * sizeof(int));
  mt.d_row_seq = (int*)put(mt.row_seq.data(), R * sizeof(int));
  mt.d_seqs = (SeqDesc*)put(mt.seqs.data(), mt.seqs.size() * sizeof(SeqDesc));
  mt.d_ctxs = (CtxDesc*)put(mt.ctxs.data(), mt.ctxs.size() * sizeof(CtxDesc));
  {
    // tensor maps over each context's K/V planes for the tcgen05 attention (its P cached rows)
    const s1_shape& s = m->sh;
    const size_t mb = attention_ctx_map_bytes();
    std::vector<uint8_t> maps(mt.ctxs.size() * mb, 0);
    if (m->nF > 0 && attention_tc_supported(s.fa_head_dim))
      for (size_t c = 0; c < mt.ctxs.size(); ++c)
        if (!attention_ctx_map(maps.data() + c * mb, mt.ctxs[c].KV, m->nF, mt.ctxs[c].P, mt.ctxs[c].cap,
                               s.fa_kv_heads, s.fa_head_dim))
          return fail(S1_ERR_CUDA, "attention tensor map encoding failed");
    mt.d_ctx_maps = put(maps.data(), maps.size());
  }
  mt.d_chunks = (ChunkDesc*)put(mt.chunks.data(), mt.chunks.size() * sizeof(ChunkDesc));
  std::vector<int> rq;
  rq.insert(rq.end(), mt.q_row.begin(), mt.q_row.end());
  rq.insert(rq.end(), mt.q_type.begin(), mt.q_type.end());
  rq.insert(rq.end(), mt.opt_off.begin(), mt.opt_off.end());
  rq.insert(rq.end(), mt.opt_ids.begin(), mt.opt_ids.end());
  int* base = (int*)put(rq.data(), rq.size() * sizeof(int));
  const size_t nq = mt.q_row.size();
  mt.d_q_row = base;
  mt.d_q_type = base + nq;
  mt.d_opt_off = base + 2 * nq;
  mt.d_opt_ids = base + 3 * nq + (nq ? 1 : 0);
  if (dest) {
    CK(cudaMemcpy(d, h, off, cudaMemcpyHostToDevice));
  } else {
    CK(cudaMemcpyAsync(d, h, off, cudaMemcpyHostToDevice, m->stream));
    CK(cudaEventRecord(m->meta_done, m->stream));
  }
  m->h2d_bytes += (long long)off;
  return S1_OK;
}

// Routes the allocations and frees of one call on a model through the model's own hooks.
struct AllocScope {
  const Alloc* prev;
  explicit AllocScope(const s1_model* m) : prev(t_alloc) { t_alloc = m ? &m->al : prev; }
  ~AllocScope() { t_alloc = prev; }
  AllocScope(const AllocScope&) = delete;
  AllocScope& operator=(const AllocScope&) = delete;
};

bool valid_model(const s1_model* m) { return m && m->magic == MODEL_MAGIC; }
bool valid_state(const s1_model* m, const s1_state* st) {
  return st && st->magic == STATE_MAGIC && st->model == m;
}

// ---------------------------------------------------------------------------------------
// GEMM dispatch
// For a residual-add GEMM, `norm_w` (may be NULL) is the weight of the RMSNorm that follows it;
// when the GEMM's split-K reduction also forms that norm (into the normed-activation buffer),
// *normed is set and the caller launches no norm of its own.
int gemm(s1_model* m, const f16* X, const f16* W, int M, int N, int K, int epi, void* out, int ldo,
         const float* norm_w = nullptr, bool* normed = nullptr) {
  ProfScope ps(m, S1_PROF_GEMM, 2.0 * M * N * K, (double)N * K * 2 + (double)M * K * 2);
  if (normed) *normed = false;
  if (m->gemm_impl == 0 && !m->force_simt && gemm_tc_supported(M, N, K, epi)) {
    LaunchCtx lc{m->stream, m->d_err, m->num_sms, &m->launches};
    if (norm_w && normed && m->fuse_norm) {
      lc.norm_w = norm_w;
      lc.norm_out = m->sc.xn;
      lc.norm_eps = m->sh.rms_eps;
      lc.norm_done = normed;
    }
    // the projection buffer is free whenever a residual-add GEMM runs (its contents were
    // consumed by the layer's mixer), so it serves as the tuning output of those shapes
    lc.tune = !m->prof;
    lc.tune_out = m->sc.proj;
    lc.tune_floats = (size_t)m->sc.rows * m->n_proj;
    lc.tune_flush = m->tune_flush;
    lc.tune_flush_bytes = m->tune_flush_bytes;
    CK(launch_gemm_tc(X, W, M, N, K, epi, out, ldo, m->sc.ws, m->sc.ws_floats, lc));
  } else {
    CK(launch_gemm_simt(X, W, M, N, K, epi, out, ldo, m->stream));
    m->launches += 1;
  }
  return S1_OK;
}

// One forward pass over the packed rows described by `mt` (metadata already uploaded):
// input rows, every decoder layer, and (if questions are present) the readout.
int run_forward(s1_model* m, Meta& mt, const bf16* d_embeds, float* probs, float* stats,
                float* hidden, bool want_lm = false) {
  const s1_shape& s = m->sh;
  const int R = (int)mt.row_src.size();
  const int nseq = (int)mt.seqs.size();
  const int d = s.d_model, F = s.ffn;
  Scratch& sc = m->sc;
  cudaStream_t st = m->stream;
  int max_keys = 0;     // longest key range of any sequence (snapshot rows + own rows)
  long att_tiles = 0;   // 64-row query tiles of the attention launches (per head)
  long att_tiles128 = 0;   // the same in 128-row tiles (the tensor-core kernel's)
  for (const SeqDesc& q : mt.seqs) {
    max_keys = std::max(max_keys, q.len + (q.ctx_in >= 0 ? mt.ctxs[q.ctx_in].P : 0));
    att_tiles += (q.len + 63) / 64;
    att_tiles128 += (q.len + 127) / 128;
  }
  const size_t plane = (size_t)R * d;
  if (m->trace && (long long)((s.n_layers + 1) * plane) > m->trace_floats)
    return fail(S1_ERR_BUDGET, "layer trace holds %lld floats, this call needs %zu", m->trace_floats,
                (size_t)(s.n_layers + 1) * plane);
  {
    ProfScope ps(m, S1_PROF_OTHER, 0, (double)R * d * 6);
    CK(launch_embed(m->embed, mt.d_row_src, d_embeds, sc.x, R, d, st));
    m->launches += 1;
  }
  if (m->trace) CK(cudaMemcpyAsync(m->trace, sc.x, plane * 4, cudaMemcpyDeviceToDevice, st));
  int li = 0;
  bool normed = false;   // xn already holds this layer's input norm (formed by the previous reduction)
  for (const Layer& L : m->layers) {
    if (!normed) {
      ProfScope ps(m, S1_PROF_NORM, 0, (double)R * d * 6);
      CK(launch_rmsnorm(sc.x, L.attn_norm, sc.xn, R, d, s.rms_eps, st));
      m->launches += 1;
    }
    int rc = gemm(m, sc.xn, L.w_in, R, L.n_in, d, EPI_F32, sc.proj, L.n_in);
    if (rc) return rc;
    if (!L.full) {
      const int H = s.la_heads;
      float* gin = sc.proj;   // the gated delta rule's input rows [q | k | v | a | b]
      if (L.conv_w) {
        // short causal convolution + SiLU of q | k | v (prefixes first when the call also
        // continues them: their snapshots' history is what the later sequences read)
        ProfScope ps(m, S1_PROF_GDN, 0, 0);
        const int split = (mt.n_first > 0 && mt.n_first < nseq) ? mt.n_first : nseq;
        const int ch = 2 * H * s.la_dk + H * s.la_dv;
        CK(launch_short_conv(sc.proj, sc.projc, L.n_in, ch, L.conv_w, s.conv_width, mt.d_seqs, 0, split, mt.max_len,
                             mt.d_ctxs, L.ord, st));
        if (split < nseq)
          CK(launch_short_conv(sc.proj, sc.projc, L.n_in, ch, L.conv_w, s.conv_width, mt.d_seqs, split, nseq - split,
                               mt.max_len, mt.d_ctxs, L.ord, st));
        m->launches += split < nseq ? 2 : 1;
        gin = sc.projc;
      }
      {
        ProfScope ps(m, S1_PROF_GDN, 0, 0);
        const int nch = (int)mt.chunks.size();
        if (!m->gdn_token && gdn_chunked_supported(H, s.la_dk, s.la_dv, L.n_in)) {
          // (the chunked path normalises q, k and forms the gates inside its first kernel)
          if ((size_t)nch > m->schunk_chunks) {
            CK(cudaStreamSynchronize(st));
            drop_graphs(m);
            dfree(m->schunk);
            const size_t cap = std::max<size_t>(nch, 2 * m->schunk_chunks);
            m->schunk = dalloc(cap * gdn_chunk_bytes(H, s.la_dk));
            m->schunk_chunks = m->schunk ? cap : 0;
            if (!m->schunk) return fail(S1_ERR_OOM, "chunk-state buffer (%zu chunks) allocation failed", cap);
          }
          const GdnBufs gb = gdn_bufs(sc.gdn, (size_t)sc.rows, m->schunk, m->schunk_chunks, H, s.la_dk);
          CK(launch_gdn_chunked(gin, L.n_in, sc.loga, s.l2_eps, sc.mix, mt.d_seqs, nseq, mt.d_chunks, nch,
                                mt.d_ctxs, L.ord, H, s.la_dk, s.la_dv, gb, mt.n_first, mt.fold_from, mt.out_fold,
                                m->d_err, m->num_sms, st, &m->launches));
        } else {
          CK(launch_gdn_prep(gin, L.n_in, sc.loga, sc.beta, R, H, s.la_dk, s.la_dv, s.l2_eps, st));
          m->launches += 1;
          const int split = (mt.n_first > 0 && mt.n_first < nseq) ? mt.n_first : nseq;
          CK(launch_gdn_scan(gin, L.n_in, sc.loga, sc.beta, sc.mix, mt.d_seqs, split, mt.d_ctxs,
                             L.ord, H, s.la_dk, s.la_dv, st));
          if (split < nseq)
            CK(launch_gdn_scan(gin, L.n_in, sc.loga, sc.beta, sc.mix, mt.d_seqs + split, nseq - split,
                               mt.d_ctxs, L.ord, H, s.la_dk, s.la_dv, st));
          m->launches += split < nseq ? 2 : 1;
        }
      }
    } else {
      {
        ProfScope ps(m, S1_PROF_OTHER, 0, 0);
        CK(launch_rope_split(sc.proj, L.n_in, m->rope_tab, mt.d_row_seq, mt.d_seqs, mt.d_ctxs, L.ord,
                             sc.q, sc.knew, sc.vnew, R, s.fa_q_heads, s.fa_kv_heads, s.fa_head_dim, st));
        m->launches += 1;
      }
      {
        ProfScope ps(m, S1_PROF_ATTN, 0, 0);
        if (m->attn_sync || !attention_tc_supported(s.fa_head_dim))
          CK(launch_attention(sc.q, sc.knew, sc.vnew, sc.mix, mt.d_seqs, nseq, mt.d_ctxs, L.ord,
                              s.fa_q_heads, s.fa_kv_heads, s.fa_head_dim, mt.max_len, max_keys,
                              att_tiles * s.fa_q_heads, m->num_sms, st));
        else
          CK(launch_attention_tc(sc.q, sc.knew, sc.vnew, sc.mix, R, mt.d_seqs, nseq, mt.d_ctxs, mt.d_ctx_maps,
                                 L.ord, s.fa_q_heads, s.fa_kv_heads, s.fa_head_dim, mt.max_len, max_keys,
                                 att_tiles128 * s.fa_q_heads, m->num_sms, m->d_err, st));
        m->launches += 1;
      }
    }
    rc = gemm(m, sc.mix, L.w_o, R, d, L.k_o, EPI_RESADD, sc.x, d, L.mlp_norm, &normed);
    if (rc) return rc;
    if (!normed) {
      ProfScope ps(m, S1_PROF_NORM, 0, (double)R * d * 6);
      CK(launch_rmsnorm(sc.x, L.mlp_norm, sc.xn, R, d, s.rms_eps, st));
      m->launches += 1;
    }
    rc = gemm(m, sc.xn, L.w_gu, R, 2 * F, d, EPI_SWIGLU, sc.h, F);
    if (rc) return rc;
    // (the last layer's output is normalised by the readout, on the question rows only)
    const float* next_norm = li + 1 < (int)m->layers.size() ? m->layers[li + 1].attn_norm : nullptr;
    rc = gemm(m, sc.h, L.w_down, R, d, F, EPI_RESADD, sc.x, d, next_norm, &normed);
    if (rc) return rc;
    ++li;
    if (m->trace) CK(cudaMemcpyAsync(m->trace + (size_t)li * plane, sc.x, plane * 4, cudaMemcpyDeviceToDevice, st));
  }
  const int nq = (int)mt.q_row.size();
  if (nq > 0) {
    ProfScope ps(m, S1_PROF_OTHER, 0, 0);
    float *hn = nullptr, *z = nullptr;
    const int no = (int)mt.opt_ids.size();
    if (want_lm) {
      const size_t need = (size_t)no + vocab_lm_scratch_floats(nq, no, d, s.vocab, m->num_sms);
      if (need > m->lm_floats) {
        CK(cudaStreamSynchronize(st));
        dfree(m->lm_buf);
        m->lm_buf = (float*)dalloc(need * 4);
        m->lm_floats = m->lm_buf ? need : 0;
        if (!m->lm_buf) return fail(S1_ERR_OOM, "log-probability scratch allocation failed");
      }
      z = m->lm_buf + no;
      hn = z + no;
    }
    CK(launch_readout(sc.x, m->final_norm, m->embed, d, s.rms_eps, mt.d_q_row, mt.d_q_type,
                      mt.d_opt_off, mt.d_opt_ids, nq, probs, stats, hidden, mt.max_opts, hn, z, st));
    m->launches += 1;
    if (want_lm) {
      LaunchCtx lc{st, m->d_err, m->num_sms, &m->launches};
      CK(launch_vocab_lm(m->embed, s.vocab, d, hn, z, mt.d_opt_off, nq, m->lm_buf, hn + (size_t)nq * d, lc,
                         !m->vocab_simt));
    }
  }
  return S1_OK;
}

int check_device_error(s1_model* m) {
  int err = 0;
  CK(cudaMemcpyAsync(&err, m->d_err, sizeof(int), cudaMemcpyDeviceToHost, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  if (err) {
    CK(cudaMemsetAsync(m->d_err, 0, sizeof(int), m->stream));
    CK(cudaStreamSynchronize(m->stream));
    return fail(S1_ERR_DEVICE_TIMEOUT, "a bounded device wait gave up (code %d)", err);
  }
  return S1_OK;
}

size_t state_S_floats(const s1_model* m) {
  return (size_t)m->nG * m->sh.la_heads * m->sh.la_dv * m->sh.la_dk;
}
size_t state_KV_elems(const s1_model* m, int cap) {
  return (size_t)m->nF * 2 * cap * m->sh.fa_kv_heads * m->sh.fa_head_dim;
}
// short-convolution history: the last width - 1 input rows of q | k | v per gated delta-rule layer
size_t state_conv_floats(const s1_model* m) {
  const s1_shape& s = m->sh;
  if (s.conv_width <= 1) return 0;
  return (size_t)m->nG * (s.conv_width - 1) * (2 * s.la_heads * s.la_dk + s.la_heads * s.la_dv);
}

int new_state(s1_model* m, int cap, s1_state** out) {
  const size_t sb = align_up(state_S_floats(m) * 4, 1024);
  const size_t kb = align_up(state_KV_elems(m, cap) * 2, 1024);
  const size_t cb = align_up(state_conv_floats(m) * 4, 1024);
  void* mem = dalloc(sb + kb + cb);
  if (!mem) return fail(S1_ERR_OOM, "state allocation (%zu bytes) failed", sb + kb + cb);
  s1_state* st = new s1_state;
  st->al = m->al;
  st->magic = STATE_MAGIC;
  st->model = m;
  st->P = 0;
  st->cap = cap;
  st->mem = mem;
  st->S = (float*)mem;
  st->KV = (f16*)((char*)mem + sb);
  st->conv = cb ? (float*)((char*)mem + sb + kb) : nullptr;
  *out = st;
  return S1_OK;
}

int validate_ids(const int32_t* ids, int n, int V, const char* what) {
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= V) return fail(S1_ERR_INVALID_ARG, "%s id %d at %d outside [0,%d)", what, ids[i], i, V);
  return S1_OK;
}

int validate_question(const s1_model* m, const s1_question& q, int idx, bool check_ids) {
  if (q.type < S1_CHOICE || q.type > S1_NOUL) return fail(S1_ERR_INVALID_ARG, "question %d: unknown type %d", idx, q.type);
  if (q.n_suffix < 1 || !q.suffix) return fail(S1_ERR_INVALID_ARG, "question %d: empty suffix", idx);
  if (!q.option_ids) return fail(S1_ERR_INVALID_ARG, "question %d: no option ids", idx);
  if (q.type == S1_CHOICE && q.n_options < 1) return fail(S1_ERR_INVALID_ARG, "question %d: choice needs >= 1 option", idx);
  if (q.type == S1_SCORE && q.n_options < 2) return fail(S1_ERR_INVALID_ARG, "question %d: score needs >= 2 levels", idx);
  if (q.type == S1_NOUL && q.n_options != 2) return fail(S1_ERR_INVALID_ARG, "question %d: noul takes exactly {yes, no}", idx);
  if (q.n_options > S1_MAX_OPTIONS) return fail(S1_ERR_BUDGET, "question %d: %d options > %d", idx, q.n_options, S1_MAX_OPTIONS);
  if (check_ids) {
    int rc = validate_ids(q.suffix, q.n_suffix, m->sh.vocab, "suffix");
    if (rc) return rc;
    rc = validate_ids(q.option_ids, q.n_options, m->sh.vocab, "option");
    if (rc) return rc;
  }
  return S1_OK;
}

// Builds the packed metadata of a decide call over n_req (state, questions) groups.
int build_decide_meta(s1_model* m, int n_req, const s1_state* const* states, const s1_question* const* qs,
                      const int32_t* n_q, bool check_ids, Meta& mt, int* total_rows, int* total_q,
                      int* total_opts) {
  int R = 0, NQ = 0, NO = 0;
  for (int r = 0; r < n_req; ++r) {
    if (!valid_state(m, states[r])) return fail(S1_ERR_INVALID_HANDLE, "state %d is not a live state of this model", r);
    if (n_q[r] < 0 || (n_q[r] > 0 && !qs[r])) return fail(S1_ERR_INVALID_ARG, "request %d: bad question array", r);
    for (int j = 0; j < n_q[r]; ++j) {
      int rc = validate_question(m, qs[r][j], j, check_ids);
      if (rc) return rc;
      if (states[r]->P + qs[r][j].n_suffix > m->max_pos) return fail(S1_ERR_BUDGET, "position budget exceeded");
      R += qs[r][j].n_suffix;
      NO += qs[r][j].n_options;
      NQ += 1;
      if (R > m->sh.max_rows) return fail(S1_ERR_BUDGET, "%d suffix rows exceed max_rows %d", R, m->sh.max_rows);
    }
  }
  if (NQ == 0) return fail(S1_ERR_INVALID_ARG, "no questions");
  int rc = ensure_scratch(m, R, NO);
  if (rc) return rc;
  mt.row_src.reserve(R);
  mt.row_seq.reserve(R);
  mt.opt_off.push_back(0);
  int row = 0;
  for (int r = 0; r < n_req; ++r) {
    const s1_state* st = states[r];
    mt.ctxs.push_back(CtxDesc{st->S, st->KV, st->P, st->cap, st->conv});
    for (int j = 0; j < n_q[r]; ++j) {
      const s1_question& q = qs[r][j];
      const int sidx = (int)mt.seqs.size();
      mt.seqs.push_back(SeqDesc{row, q.n_suffix, st->P, r, -1, 0});
      mt.max_len = std::max(mt.max_len, q.n_suffix);
      for (int i = 0; i < q.n_suffix; ++i) {
        mt.row_src.push_back(check_ids ? q.suffix[i] : 0);
        mt.row_seq.push_back(sidx);
      }
      mt.q_row.push_back(row + q.n_suffix - 1);
      mt.q_type.push_back(q.type);
      for (int o = 0; o < q.n_options; ++o) mt.opt_ids.push_back(check_ids ? q.option_ids[o] : 0);
      mt.opt_off.push_back(mt.opt_off.back() + q.n_options);
      mt.max_opts = std::max(mt.max_opts, q.n_options);
      row += q.n_suffix;
    }
  }
  *total_rows = R;
  *total_q = NQ;
  *total_opts = NO;
  return S1_OK;
}

int build_prefill_meta(s1_model* m, int n_req, const int32_t* n_tokens, const int32_t* n_embeds,
                       s1_state* const* states, Meta& mt, int* total_rows, int* total_embeds) {
  int R = 0, NE = 0;
  for (int r = 0; r < n_req; ++r) {
    const int P = n_tokens[r] + n_embeds[r];
    if (n_tokens[r] < 0 || n_embeds[r] < 0 || P < 1) return fail(S1_ERR_INVALID_ARG, "request %d: empty prefix", r);
    if (P > states[r]->cap) return fail(S1_ERR_BUDGET, "request %d: prefix %d rows > state capacity %d", r, P, states[r]->cap);
    if (P > m->max_pos) return fail(S1_ERR_BUDGET, "position budget exceeded");
    R += P;
    NE += n_embeds[r];
    if (R > m->sh.max_rows) return fail(S1_ERR_BUDGET, "%d prefix rows exceed max_rows %d", R, m->sh.max_rows);
  }
  int rc = ensure_scratch(m, R);
  if (rc) return rc;
  int row = 0, erow = 0;
  for (int r = 0; r < n_req; ++r) {
    const int P = n_tokens[r] + n_embeds[r];
    mt.ctxs.push_back(CtxDesc{states[r]->S, states[r]->KV, 0, states[r]->cap, states[r]->conv});
    mt.seqs.push_back(SeqDesc{row, P, 0, -1, r, 0});
    mt.max_len = std::max(mt.max_len, P);
    for (int i = 0; i < P; ++i) mt.row_seq.push_back(r);
    for (int i = 0; i < n_embeds[r]; ++i) mt.row_src.push_back(-1 - (erow + i));
    for (int i = 0; i < n_tokens[r]; ++i) mt.row_src.push_back(0);  // filled by the caller
    erow += n_embeds[r];
    row += P;
  }
  *total_rows = R;
  *total_embeds = NE;
  return S1_OK;
}

}  // namespace

// =======================================================================================
// C ABI
extern "C" {

const char* s1_last_error(void) { return g_err.c_str(); }

int s1_split_prefix(const int32_t* const* streams, const int32_t* lens, int32_t n, int32_t min_suffix,
                    int32_t align, int32_t* prefix_len) {
  if (n < 1 || !streams || !lens || !prefix_len) return fail(S1_ERR_INVALID_ARG, "split: bad arguments");
  if (min_suffix < 1) return fail(S1_ERR_INVALID_ARG, "split: min_suffix must be >= 1");
  int32_t cap = INT32_MAX;
  for (int i = 0; i < n; ++i) {
    if (!streams[i] || lens[i] < min_suffix) return fail(S1_ERR_INVALID_ARG, "split: stream %d shorter than min_suffix", i);
    cap = std::min(cap, lens[i] - min_suffix);
  }
  int32_t P = 0;
  while (P < cap) {
    const int32_t t = streams[0][P];
    bool same = true;
    for (int i = 1; i < n && same; ++i) same = streams[i][P] == t;
    if (!same) break;
    ++P;
  }
  if (align > 1) P -= P % align;
  *prefix_len = P;
  return S1_OK;
}
const char* s1_version(void) { return "s1 0.1 (sm_103a)"; }

int s1_set_allocator(void* (*alloc)(size_t, void*), void (*free_fn)(void*, void*), void* ctx) {
  if ((alloc == nullptr) != (free_fn == nullptr)) return fail(S1_ERR_INVALID_ARG, "alloc and free must both be set or both NULL");
  g_al.alloc = alloc;
  g_al.free = free_fn;
  g_al.ctx = ctx;
  return S1_OK;
}

int s1_model_create(const s1_shape* shape, const s1_weights* w, s1_model** out) {
  if (!shape || !w || !out) return fail(S1_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  const s1_shape& s = *shape;
  if (s.vocab <= 0 || s.d_model <= 0 || s.n_layers <= 0 || s.ffn <= 0 || !s.layer_is_full)
    return fail(S1_ERR_INVALID_ARG, "shape: non-positive size or missing layer kinds");
  if (s.d_model % 64 || s.ffn % 64) return fail(S1_ERR_INVALID_ARG, "shape: d_model and ffn must be multiples of 64");
  if (s.weight_dtype != S1_F32 && s.weight_dtype != S1_BF16) return fail(S1_ERR_INVALID_ARG, "shape: weight_dtype");
  if (s.lora_rank < 0 || s.lora_rank > 1024) return fail(S1_ERR_INVALID_ARG, "shape: lora_rank");
  if (!(s.rms_eps >= 0) || !(s.l2_eps >= 0) || !(s.rope_theta > 0)) return fail(S1_ERR_INVALID_ARG, "shape: eps/theta");
  int nG = 0, nF = 0;
  for (int l = 0; l < s.n_layers; ++l) (s.layer_is_full[l] ? nF : nG)++;
  if (nG && (s.la_heads <= 0 || s.la_dk != s.la_dv || (s.la_dk != 64 && s.la_dk != 128)))
    return fail(S1_ERR_UNSUPPORTED, "gated delta-rule layers need la_dk == la_dv in {64, 128}");
  if (nF && (s.fa_q_heads <= 0 || s.fa_kv_heads <= 0 || s.fa_q_heads % s.fa_kv_heads ||
             (s.fa_head_dim != 64 && s.fa_head_dim != 128)))
    return fail(S1_ERR_UNSUPPORTED, "attention layers need Hq %% Hkv == 0 and head_dim in {64, 128}");
  if (s.conv_width < 0 || s.conv_width > 8) return fail(S1_ERR_INVALID_ARG, "shape: conv_width outside [0, 8]");
  if (!w->embed || !w->final_norm || !w->layer) return fail(S1_ERR_INVALID_ARG, "weights: NULL tensor array");

  s1_model* m = new s1_model();
  m->al = g_al;
  AllocScope alloc_scope(m);
  m->magic = MODEL_MAGIC;
  m->sh = s;
  m->is_full.assign(s.layer_is_full, s.layer_is_full + s.n_layers);
  m->sh.layer_is_full = m->is_full.data();
  if (m->sh.max_rows <= 0) m->sh.max_rows = 32768;
  m->nG = nG;
  m->nF = nF;
  const int d = s.d_model, F = s.ffn;
  const int H = s.la_heads, Dk = s.la_dk, Dv = s.la_dv;
  const int Hq = s.fa_q_heads, Hkv = s.fa_kv_heads, hd = s.fa_head_dim;
  // packed in-projection widths, rounded up to whole 32-column groups (the tensor-core GEMM's
  // N granule) with zero weight rows; the padding columns of the projection are never read
  const int in_gdn = 2 * H * Dk + H * Dv + 2 * H, in_fa = (Hq + 2 * Hkv) * hd;
  m->n_in_gdn = nG ? (in_gdn + 31) / 32 * 32 : 0;
  m->n_in_fa = nF ? (in_fa + 31) / 32 * 32 : 0;
  m->n_proj = std::max(m->n_in_gdn, m->n_in_fa);
  m->n_mix = std::max(nG ? H * Dv : 0, nF ? Hq * hd : 0);
  const char* gi = getenv("S1_GEMM");
  m->force_simt = gi && strcmp(gi, "simt") == 0;
  const char* gd = getenv("S1_GDN");
  m->gdn_token = gd && strcmp(gd, "token") == 0;
  const char* gv = getenv("S1_VOCAB");
  m->vocab_simt = gv && strcmp(gv, "simt") == 0;
  const char* ga = getenv("S1_ATTN");
  m->attn_sync = ga && strcmp(ga, "sync") == 0;
  const char* nf = getenv("S1_NORM_FUSE");
  m->fuse_norm = !(nf && strcmp(nf, "0") == 0);
  m->gemm_impl = m->force_simt ? 1 : 0;
  auto bail = [&](int rc) {
    s1_model_destroy(m);
    return rc;
  };
  if (cudaGetDevice(&m->device) != cudaSuccess) return bail(fail(S1_ERR_CUDA, "no CUDA device"));
  cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
  if (cudaEventCreateWithFlags(&m->meta_done, cudaEventDisableTiming) != cudaSuccess)
    return bail(fail(S1_ERR_CUDA, "event creation failed"));
  cudaEventRecord(m->meta_done, m->stream);

  // ---- weight arena
  std::vector<size_t> offs;
  size_t total = 0;
  auto reserve = [&](size_t bytes) {
    offs.push_back(total);
    total += align_up(bytes, 1024);
    return offs.size() - 1;
  };
  const size_t i_embed = reserve((size_t)s.vocab * d * 2);
  const size_t i_fnorm = reserve((size_t)d * 4);
  std::vector<size_t> li(s.n_layers * 7);
  const int conv_ch = 2 * H * Dk + H * Dv;   // channels of the short convolution (q | k | v)
  for (int l = 0; l < s.n_layers; ++l) {
    const bool full = m->is_full[l];
    const int n_in = full ? m->n_in_fa : m->n_in_gdn;
    const int k_o = full ? Hq * hd : H * Dv;
    li[l * 7 + 0] = reserve((size_t)d * 4);
    li[l * 7 + 1] = reserve((size_t)d * 4);
    li[l * 7 + 2] = reserve((size_t)n_in * d * 2);
    li[l * 7 + 3] = reserve((size_t)d * k_o * 2);
    li[l * 7 + 4] = reserve((size_t)2 * F * d * 2);
    li[l * 7 + 5] = reserve((size_t)d * F * 2);
    li[l * 7 + 6] = reserve(!full && s.conv_width > 0 ? (size_t)conv_ch * s.conv_width * 4 : 0);
  }
  m->arena = dalloc(total);
  if (!m->arena) return bail(fail(S1_ERR_OOM, "weight arena (%zu bytes) allocation failed", total));
  char* A = (char*)m->arena;
  m->embed = (f16*)(A + offs[i_embed]);
  m->final_norm = (float*)(A + offs[i_fnorm]);
  int ordG = 0, ordF = 0;
  for (int l = 0; l < s.n_layers; ++l) {
    Layer L;
    L.full = m->is_full[l];
    L.ord = L.full ? ordF++ : ordG++;
    L.attn_norm = (float*)(A + offs[li[l * 7 + 0]]);
    L.mlp_norm = (float*)(A + offs[li[l * 7 + 1]]);
    L.w_in = (f16*)(A + offs[li[l * 7 + 2]]);
    L.n_in = L.full ? m->n_in_fa : m->n_in_gdn;
    L.w_o = (f16*)(A + offs[li[l * 7 + 3]]);
    L.k_o = L.full ? Hq * hd : H * Dv;
    L.w_gu = (f16*)(A + offs[li[l * 7 + 4]]);
    L.w_down = (f16*)(A + offs[li[l * 7 + 5]]);
    L.conv_w = (!L.full && s.conv_width > 0) ? (float*)(A + offs[li[l * 7 + 6]]) : nullptr;
    m->layers.push_back(L);
  }

  // ---- upload + merge, one tensor at a time through a staging buffer
  const int wb = s.weight_dtype == S1_BF16;
  const size_t esz = wb ? 2 : 4;
  const int r = s.lora_rank;
  size_t max_numel = (size_t)s.vocab * d;
  for (int l = 0; l < s.n_layers; ++l) max_numel = std::max(max_numel, (size_t)F * d);
  max_numel = std::max(max_numel, (size_t)m->n_proj * d);
  const size_t lora_numel = r > 0 ? (size_t)r * std::max(std::max(d, F), std::max(m->n_proj, m->n_mix)) : 0;
  char* stage = (char*)dalloc(max_numel * esz + 2 * lora_numel * esz + 4096);
  if (!stage) return bail(fail(S1_ERR_OOM, "staging allocation failed"));
  char* stA = stage + align_up(max_numel * esz, 256);
  char* stB = stA + align_up(lora_numel * esz, 256);
  int rc = S1_OK;
  auto up = [&](const void* host, size_t numel, void* dev) -> int {
    if (!host) return fail(S1_ERR_INVALID_ARG, "weights: NULL tensor");
    CK(cudaMemcpy(dev, host, numel * esz, cudaMemcpyHostToDevice));
    return S1_OK;
  };
  // base matrix [out_f, in_f] (+ optional LoRA pair) -> f16 at dst
  auto merge = [&](const void* Wh, int out_f, int in_f, int l, int target, f16* dst, int row0,
                   int inter, int half) -> int {
    int rc2 = up(Wh, (size_t)out_f * in_f, stage);
    if (rc2) return rc2;
    const void* Ad = nullptr;
    const void* Bd = nullptr;
    int rank = 0;
    if (r > 0 && target >= 0 && w->lora_a && w->lora_b && w->lora_a[l * 7 + target] && w->lora_b[l * 7 + target]) {
      rc2 = up(w->lora_a[l * 7 + target], (size_t)r * in_f, stA);
      if (rc2) return rc2;
      rc2 = up(w->lora_b[l * 7 + target], (size_t)out_f * r, stB);
      if (rc2) return rc2;
      Ad = stA;
      Bd = stB;
      rank = r;
    }
    const float scale = r > 0 ? s.lora_alpha / (float)r : 0.f;
    CK(launch_merge_lora(stage, wb, Ad, Bd, wb, rank, scale, out_f, in_f, dst, row0, inter, half, F,
                         nullptr, nullptr, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    return S1_OK;
  };
  auto to_f32 = [&](const void* host, size_t n, float* dst) -> int {
    int rc2 = up(host, n, stage);
    if (rc2) return rc2;
    CK(launch_to_f32(stage, wb, dst, n, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    return S1_OK;
  };
  auto norm = [&](const void* host, float* dst) -> int { return to_f32(host, d, dst); };
  rc = merge(w->embed, s.vocab, d, 0, -1, m->embed, 0, 0, 0);
  if (!rc) rc = norm(w->final_norm, m->final_norm);
  size_t t = 0;
  for (int l = 0; l < s.n_layers && !rc; ++l) {
    Layer& L = m->layers[l];
    const void* const* T = w->layer + t;
    if (!L.full) {
      t += s.conv_width > 0 ? 12 : 11;
      rc = norm(T[0], L.attn_norm);
      if (!rc) rc = merge(T[1], H * Dk, d, l, 0, L.w_in, 0, 0, 0);
      if (!rc) rc = merge(T[2], H * Dk, d, l, 1, L.w_in, H * Dk, 0, 0);
      if (!rc) rc = merge(T[3], H * Dv, d, l, 2, L.w_in, 2 * H * Dk, 0, 0);
      if (!rc) rc = merge(T[4], H, d, l, -1, L.w_in, 2 * H * Dk + H * Dv, 0, 0);
      if (!rc) rc = merge(T[5], H, d, l, -1, L.w_in, 2 * H * Dk + H * Dv + H, 0, 0);
      if (!rc) rc = merge(T[6], d, H * Dv, l, 3, L.w_o, 0, 0, 0);
      if (!rc) rc = norm(T[7], L.mlp_norm);
      if (!rc) rc = merge(T[8], F, d, l, 4, L.w_gu, 0, 1, 0);
      if (!rc) rc = merge(T[9], F, d, l, 5, L.w_gu, 0, 1, 1);
      if (!rc) rc = merge(T[10], d, F, l, 6, L.w_down, 0, 0, 0);
      if (!rc && L.conv_w) rc = to_f32(T[11], (size_t)conv_ch * s.conv_width, L.conv_w);
    } else {
      t += 9;
      rc = norm(T[0], L.attn_norm);
      if (!rc) rc = merge(T[1], Hq * hd, d, l, 0, L.w_in, 0, 0, 0);
      if (!rc) rc = merge(T[2], Hkv * hd, d, l, 1, L.w_in, Hq * hd, 0, 0);
      if (!rc) rc = merge(T[3], Hkv * hd, d, l, 2, L.w_in, (Hq + Hkv) * hd, 0, 0);
      if (!rc) rc = merge(T[4], d, Hq * hd, l, 3, L.w_o, 0, 0, 0);
      if (!rc) rc = norm(T[5], L.mlp_norm);
      if (!rc) rc = merge(T[6], F, d, l, 4, L.w_gu, 0, 1, 0);
      if (!rc) rc = merge(T[7], F, d, l, 5, L.w_gu, 0, 1, 1);
      if (!rc) rc = merge(T[8], d, F, l, 6, L.w_down, 0, 0, 0);
    }
  }
  dfree(stage);
  if (rc) return bail(rc);
  for (const Layer& L : m->layers) {
    const int used = L.full ? in_fa : in_gdn;
    if (L.n_in > used &&
        cudaMemsetAsync(L.w_in + (size_t)used * d, 0, (size_t)(L.n_in - used) * d * 2, m->stream) != cudaSuccess)
      return bail(fail(S1_ERR_CUDA, "in-projection padding rows: memset failed"));
  }

  // ---- rotary table, error word
  m->max_pos = 2 * m->sh.max_rows;
  if (nF) {
    m->rope_tab = (float2*)dalloc((size_t)m->max_pos * (hd / 2) * sizeof(float2));
    if (!m->rope_tab) return bail(fail(S1_ERR_OOM, "rope table allocation failed"));
    if (launch_rope_table(m->rope_tab, m->max_pos, hd, (double)s.rope_theta, m->stream) != cudaSuccess)
      return bail(fail(S1_ERR_CUDA, "rope table kernel failed"));
  }
  m->d_err = (int*)dalloc(256);
  if (!m->d_err) return bail(fail(S1_ERR_OOM, "error word allocation failed"));
  // The GEMM autotuner times each candidate tile from a flushed L2 (a write larger than L2
  // before each run); the buffer comes from the model's allocator like all its device memory.
  {
    const char* tn = getenv("S1_GEMM_TUNE");
    if (!(tn && tn[0] == '0')) {
      m->tune_flush_bytes = (size_t)192 << 20;
      m->tune_flush = dalloc(m->tune_flush_bytes);
      if (!m->tune_flush) return bail(fail(S1_ERR_OOM, "autotuner L2-flush buffer allocation failed"));
    }
  }
  if (cudaMemsetAsync(m->d_err, 0, 256, m->stream) != cudaSuccess ||
      cudaStreamSynchronize(m->stream) != cudaSuccess)
    return bail(fail(S1_ERR_CUDA, "model initialisation failed: %s", cudaGetErrorString(cudaGetLastError())));
  *out = m;
  return S1_OK;
}

void s1_model_destroy(s1_model* m) {
  if (!valid_model(m)) return;
  AllocScope alloc_scope(m);
  cudaStreamSynchronize(m->stream);
  if (m->prof) --pdl_suppressed();
  drop_graphs(m);
  free_scratch(m->sc);
  dfree(m->arena);
  dfree(m->rope_tab);
  dfree(m->d_err);
  dfree(m->schunk);
  dfree(m->lm_buf);
  dfree(m->tune_flush);
  if (m->pinned) cudaFreeHost(m->pinned);
  if (m->meta_done) cudaEventDestroy(m->meta_done);
  for (cudaEvent_t e : m->ev_pool) cudaEventDestroy(e);
  m->magic = DEAD;
  delete m;
}

int s1_set_stream(s1_model* m, void* stream) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  CK(cudaStreamSynchronize(m->stream));
  m->stream = (cudaStream_t)stream;
  return S1_OK;
}

int s1_sync(s1_model* m) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  CK(cudaStreamSynchronize(m->stream));
  return check_device_error(m);
}

int s1_state_create(s1_model* m, int32_t capacity_rows, s1_state** out) {
  if (!valid_model(m) || !out) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (capacity_rows < 1 || capacity_rows > m->sh.max_rows) return fail(S1_ERR_BUDGET, "capacity %d outside [1, max_rows]", capacity_rows);
  return new_state(m, capacity_rows, out);
}

void s1_state_destroy(s1_state* st) {
  if (!st || st->magic != STATE_MAGIC) return;
  if (st->model && valid_model(st->model)) cudaStreamSynchronize(st->model->stream);
  {
    const Alloc* prev = t_alloc;
    t_alloc = &st->al;
    dfree(st->mem);
    t_alloc = prev;
  }
  st->magic = DEAD;
  delete st;
}

int s1_state_rows(const s1_state* st) { return (st && st->magic == STATE_MAGIC) ? st->P : -1; }

extern "C++" {
// -- CUDA graphs of the stream-ordered calls ----------------------------------------------
// Runs `body` (everything a call enqueues after its metadata upload) eagerly, or, with `cap`,
// captures it into cap->exec and launches that graph once. Kernel launches counted while
// capturing are booked to the graph, which adds them on every replay.
template <class Body>
static int run_captured(s1_model* m, s1_model::Graph* cap, Body&& body) {
  if (!cap) return body();
  const long launches0 = m->launches;
  CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
  int rc = body();
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(m->stream, &g);
  if (rc == S1_OK && ec != cudaSuccess) rc = fail(S1_ERR_CUDA, "graph capture: %s", cudaGetErrorString(ec));
  if (rc == S1_OK) {
    const cudaError_t ei = cudaGraphInstantiate(&cap->exec, g, 0);
    if (ei != cudaSuccess) rc = fail(S1_ERR_CUDA, "graph instantiation: %s", cudaGetErrorString(ei));
  }
  if (g) cudaGraphDestroy(g);
  cap->launches = m->launches - launches0;
  m->launches = launches0;
  if (rc == S1_OK) {
    CK(cudaGraphLaunch(cap->exec, m->stream));
    m->launches += cap->launches;
  }
  return rc;
}

// Signature of a stream-ordered call: every pointer, size and descriptor it passes, plus the
// state buffers it reads or writes. Two calls with equal signatures enqueue identical work.
struct CallKey {
  std::string s;
  explicit CallKey(char kind) : s(1, kind) {}
  template <class T> CallKey& add(const T& v) {
    s.append((const char*)&v, sizeof(T));
    return *this;
  }
  CallKey& state(const s1_state* st, bool with_rows) {
    add(st).add(st->S).add(st->KV).add(st->cap);
    if (with_rows) add(st->P);
    return *this;
  }
  // field by field: the struct's padding bytes are not part of the signature
  CallKey& question(const s1_question& q) {
    return add(q.type).add(q.suffix).add(q.n_suffix).add(q.option_ids).add(q.n_options);
  }
};

// With graphs on, a call whose signature was seen before replays (on its second occurrence,
// captures) a graph; `run(cap)` performs the call, capturing into `cap` when it is non-null,
// and `replayed()` applies the host-side effects of a replay. Anything else runs eagerly.
template <class Run, class Replayed>
static int graph_call(s1_model* m, const CallKey& key, Run&& run, Replayed&& replayed) {
  if (!m->graphs || m->prof || m->trace || m->stream == nullptr) return run(nullptr);
  auto it = m->graph_cache.find(key.s);
  if (it != m->graph_cache.end()) {
    CK(cudaGraphLaunch(it->second.exec, m->stream));
    m->launches += it->second.launches;
    replayed();
    return S1_OK;
  }
  if (m->graph_cache.size() >= s1_model::kMaxGraphs) return run(nullptr);
  if (m->graph_seen.size() >= s1_model::kMaxSeen) m->graph_seen.clear();
  if (m->graph_seen.insert(key.s).second) return run(nullptr);
  s1_model::Graph g;
  const int rc = run(&g);
  if (rc == S1_OK) {
    m->graph_cache[key.s] = g;
  } else {
    // an error inside the capture may have left it open: close it and drop the partial graph
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(m->stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone) {
      cudaGraph_t partial = nullptr;
      cudaStreamEndCapture(m->stream, &partial);
      if (partial) cudaGraphDestroy(partial);
    }
    cudaGetLastError();
    if (g.exec) cudaGraphExecDestroy(g.exec);
    dfree(g.meta);
  }
  return rc;
}

}  // extern "C++"

// -- prefill -----------------------------------------------------------------------------
static int prefill_impl(s1_model* m, int n_req, const int32_t* const* tokens, const int32_t* n_tokens,
                        const void* const* embeds, const int32_t* n_embeds, s1_state** states,
                        bool device_ptrs, s1_model::Graph* cap = nullptr) {
  Meta mt;
  int R = 0, NE = 0;
  int rc = build_prefill_meta(m, n_req, n_tokens, n_embeds, states, mt, &R, &NE);
  if (rc) return rc;
  // token ids: host -> pinned metadata (validated), or device -> gathered by a copy
  int row = 0;
  for (int r = 0; r < n_req; ++r) {
    row += n_embeds[r];
    if (n_tokens[r] > 0) {
      if (!tokens || !tokens[r]) return fail(S1_ERR_INVALID_ARG, "request %d: NULL tokens", r);
      if (!device_ptrs) {
        rc = validate_ids(tokens[r], n_tokens[r], m->sh.vocab, "token");
        if (rc) return rc;
        memcpy(&mt.row_src[row], tokens[r], n_tokens[r] * sizeof(int));
      }
    }
    row += n_tokens[r];
  }
  for (int r = 0; r < n_req; ++r)
    if (n_embeds[r] > 0 && (!embeds || !embeds[r])) return fail(S1_ERR_INVALID_ARG, "request %d: NULL embeds", r);
  rc = upload_meta(m, mt, cap ? &cap->meta : nullptr);
  if (rc) return rc;
  rc = run_captured(m, cap, [&]() -> int {
    if (device_ptrs) {
      int rr = 0;
      for (int r = 0; r < n_req; ++r) {
        rr += n_embeds[r];
        if (n_tokens[r] > 0)
          CK(cudaMemcpyAsync(mt.d_row_src + rr, tokens[r], n_tokens[r] * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
        rr += n_tokens[r];
      }
    }
    // given embedding rows are staged in the normed-activation buffer (free until layer 0)
    const size_t rowb = (size_t)m->sh.d_model * 2;
    if (NE > 0) {
      size_t eoff = 0;
      for (int r = 0; r < n_req; ++r) {
        if (n_embeds[r] == 0) continue;
        CK(cudaMemcpyAsync((char*)m->sc.xn + eoff, embeds[r], n_embeds[r] * rowb,
                           device_ptrs ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, m->stream));
        if (!device_ptrs) m->h2d_bytes += (long long)(n_embeds[r] * rowb);
        eoff += n_embeds[r] * rowb;
      }
    }
    return run_forward(m, mt, reinterpret_cast<const bf16*>(m->sc.xn), nullptr, nullptr, nullptr);
  });
  if (rc) return rc;
  for (int r = 0; r < n_req; ++r) states[r]->P = n_tokens[r] + n_embeds[r];
  return S1_OK;
}

int s1_prefill_state_batch(s1_model* m, int32_t n_req, const int32_t* const* tokens, const int32_t* n_tokens,
                           const void* const* embeds, const int32_t* n_embeds, s1_state** out) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (n_req < 1 || !n_tokens || !out) return fail(S1_ERR_INVALID_ARG, "bad batch arguments");
  std::vector<int32_t> ne(n_req, 0);
  if (n_embeds) ne.assign(n_embeds, n_embeds + n_req);
  std::vector<s1_state*> sts(n_req, nullptr);
  auto cleanup = [&](int rc) {
    for (s1_state* s : sts) s1_state_destroy(s);
    return rc;
  };
  for (int r = 0; r < n_req; ++r) {
    const int P = n_tokens[r] + ne[r];
    if (P < 1) return cleanup(fail(S1_ERR_INVALID_ARG, "request %d: empty prefix", r));
    if (P > m->sh.max_rows) return cleanup(fail(S1_ERR_BUDGET, "request %d: prefix %d > max_rows", r, P));
    int rc = new_state(m, P, &sts[r]);
    if (rc) return cleanup(rc);
  }
  int rc = prefill_impl(m, n_req, tokens, n_tokens, embeds, ne.data(), sts.data(), false);
  if (!rc) rc = s1_sync(m);
  if (rc) return cleanup(rc);
  for (int r = 0; r < n_req; ++r) out[r] = sts[r];
  return S1_OK;
}

int s1_prefill_state(s1_model* m, const int32_t* tokens, int32_t n_tokens, const void* embeds,
                     int32_t n_embeds, s1_state** out) {
  const void* e[1] = {embeds};
  return s1_prefill_state_batch(m, 1, &tokens, &n_tokens, e, &n_embeds, out);
}

int s1_prefill_async(s1_model* m, s1_state* st, const int32_t* d_tokens, int32_t n_tokens,
                     const void* d_embeds, int32_t n_embeds) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (!valid_state(m, st)) return fail(S1_ERR_INVALID_HANDLE, "invalid state");
  const void* e[1] = {d_embeds};
  CallKey key('P');
  key.state(st, false).add(d_tokens).add(n_tokens).add(d_embeds).add(n_embeds);
  return graph_call(
      m, key,
      [&](s1_model::Graph* cap) { return prefill_impl(m, 1, &d_tokens, &n_tokens, e, &n_embeds, &st, true, cap); },
      [&]() { st->P = n_tokens + n_embeds; });
}

// -- decide ------------------------------------------------------------------------------
static int decide_impl(s1_model* m, int n_req, const s1_state* const* states, const s1_question* const* qs,
                       const int32_t* n_q, bool device_ptrs, float* d_probs, float* d_stats,
                       float* d_hidden, Meta& mt, int* NQ, int* NO, s1_model::Graph* cap = nullptr) {
  int R = 0;
  int rc = build_decide_meta(m, n_req, states, qs, n_q, !device_ptrs, mt, &R, NQ, NO);
  if (rc) return rc;
  rc = upload_meta(m, mt, cap ? &cap->meta : nullptr);
  if (rc) return rc;
  return run_captured(m, cap, [&]() -> int {
    if (device_ptrs) {
      // gather ids from the caller's device arrays into the uploaded metadata
      int row = 0, opt = 0;
      for (int r = 0; r < n_req; ++r)
        for (int j = 0; j < n_q[r]; ++j) {
          const s1_question& q = qs[r][j];
          CK(cudaMemcpyAsync(mt.d_row_src + row, q.suffix, q.n_suffix * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
          CK(cudaMemcpyAsync(mt.d_opt_ids + opt, q.option_ids, q.n_options * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
          row += q.n_suffix;
          opt += q.n_options;
        }
    }
    return run_forward(m, mt, nullptr, d_probs, d_stats, d_hidden);
  });
}

// Copies the readout outputs (probs | stats | hidden in the scratch output block) back into
// the caller's result structs. Blocking.
static bool wants_lm(int n_req, const int32_t* n_q, s1_result* const* out) {
  for (int r = 0; r < n_req; ++r)
    for (int j = 0; j < n_q[r]; ++j)
      if (out[r] && out[r][j].lm_logprobs) return true;
  return false;
}

static int fetch_results(s1_model* m, int n_req, const s1_question* const* qs, const int32_t* n_q, int NQ, int NO,
                         bool want_hidden, s1_result* const* out, float* const* last_hidden) {
  std::vector<float> lmh;
  const bool want_lm = wants_lm(n_req, n_q, out);
  if (want_lm) {
    lmh.resize(NO);
    CK(cudaMemcpyAsync(lmh.data(), m->lm_buf, (size_t)NO * 4, cudaMemcpyDeviceToHost, m->stream));
    m->d2h_bytes += (long long)NO * 4;
  }
  float* probs = m->sc.out;
  float* stats = probs + align_up(NO, 64);
  float* hidden = stats + align_up((size_t)NQ * S1_STAT_COUNT, 64);
  const size_t nfl = (size_t)(hidden - probs) + (want_hidden ? (size_t)NQ * m->sh.d_model : 0);
  std::vector<float> h(nfl);
  CK(cudaMemcpyAsync(h.data(), probs, nfl * 4, cudaMemcpyDeviceToHost, m->stream));
  m->d2h_bytes += (long long)(nfl * 4);
  int rc = s1_sync(m);
  if (rc) return rc;
  const float* hp = h.data();
  const float* hs = hp + (stats - probs);
  const float* hh = hp + (hidden - probs);
  int qi = 0, oi = 0;
  for (int r = 0; r < n_req; ++r)
    for (int j = 0; j < n_q[r]; ++j, ++qi) {
      const int n = qs[r][j].n_options;
      s1_result& res = out[r][j];
      if (res.probs) memcpy(res.probs, hp + oi, n * 4);
      const float* sv = hs + (size_t)qi * S1_STAT_COUNT;
      res.argmax = (int32_t)sv[S1_STAT_ARGMAX];
      res.expected_score = sv[S1_STAT_EXPECTED];
      res.yes_prob = sv[S1_STAT_YES];
      res.answer_confidence = sv[S1_STAT_ANSWER_CONF];
      res.confidence = sv[S1_STAT_CONF];
      res.entropy_confidence = sv[S1_STAT_ENTROPY_CONF];
      if (want_hidden && last_hidden[r])
        memcpy(last_hidden[r] + (size_t)j * m->sh.d_model, hh + (size_t)qi * m->sh.d_model, m->sh.d_model * 4);
      if (want_lm && res.lm_logprobs) memcpy(res.lm_logprobs, lmh.data() + oi, n * 4);
      oi += n;
    }
  return S1_OK;
}

static void output_slots(s1_model* m, int NQ, int NO, float** probs, float** stats, float** hidden) {
  *probs = m->sc.out;
  *stats = *probs + align_up(NO, 64);
  *hidden = *stats + align_up((size_t)NQ * S1_STAT_COUNT, 64);
}

int s1_decide_batch(s1_model* m, int32_t n_req, const s1_state* const* states, const s1_question* const* qs,
                    const int32_t* n_q, s1_result* const* out, float* const* last_hidden) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (n_req < 1 || !states || !qs || !n_q || !out) return fail(S1_ERR_INVALID_ARG, "bad batch arguments");
  for (int r = 0; r < n_req; ++r)
    if (n_q[r] > 0 && !out[r]) return fail(S1_ERR_INVALID_ARG, "request %d: NULL results", r);
  Meta mt;
  int NQ = 0, NO = 0, R = 0;
  int rc = build_decide_meta(m, n_req, states, qs, n_q, true, mt, &R, &NQ, &NO);
  if (rc) return rc;
  float *probs, *stats, *hidden;
  output_slots(m, NQ, NO, &probs, &stats, &hidden);
  bool want_hidden = false;
  if (last_hidden)
    for (int r = 0; r < n_req; ++r) want_hidden |= (last_hidden[r] != nullptr);
  rc = upload_meta(m, mt);
  if (rc) return rc;
  rc = run_forward(m, mt, nullptr, probs, stats, want_hidden ? hidden : nullptr, wants_lm(n_req, n_q, out));
  if (rc) return rc;
  return fetch_results(m, n_req, qs, n_q, NQ, NO, want_hidden, out, last_hidden);
}

int s1_decide(s1_model* m, const s1_state* st, const s1_question* qs, int32_t n_q, s1_result* out,
              float* last_hidden) {
  return s1_decide_batch(m, 1, &st, &qs, &n_q, &out, &last_hidden);
}

int s1_decide_async(s1_model* m, const s1_state* st, const s1_question* qs_dev, int32_t n_q,
                    float* d_probs, float* d_stats, float* d_last_hidden) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (!d_probs || !d_stats) return fail(S1_ERR_INVALID_ARG, "NULL output");
  if (!valid_state(m, st)) return fail(S1_ERR_INVALID_HANDLE, "invalid state");
  if (n_q < 1 || !qs_dev) return fail(S1_ERR_INVALID_ARG, "no questions");
  CallKey key('D');
  key.state(st, true).add(d_probs).add(d_stats).add(d_last_hidden).add(n_q);
  for (int j = 0; j < n_q; ++j) key.question(qs_dev[j]);
  return graph_call(
      m, key,
      [&](s1_model::Graph* cap) {
        Meta mt;
        int NQ = 0, NO = 0;
        return decide_impl(m, 1, &st, &qs_dev, &n_q, true, d_probs, d_stats, d_last_hidden, mt, &NQ, &NO, cap);
      },
      []() {});
}

// -- fused sweep: prefixes and their questions in one pass over the layers ---------------
// Rows: every prefix, then every question suffix. Each layer's projections run once over all
// rows (the weights are streamed once per request instead of once per call); the gated
// delta-rule state pass runs the prefixes first and then the suffixes, which continue from
// the snapshot written moments before in the same layer; suffix queries read the prefix K/V
// that the same layer's RoPE step has just cached.
static int fused_impl(s1_model* m, int n_req, const int32_t* const* tokens, const int32_t* n_tokens,
                      const void* const* embeds, const int32_t* n_embeds, s1_state* const* states,
                      const s1_question* const* qs, const int32_t* n_q, bool device_ptrs, float* d_probs,
                      float* d_stats, float* d_hidden, int* NQ_out, int* NO_out, bool want_lm = false,
                      s1_model::Graph* cap = nullptr) {
  int Rp = 0, Rs = 0, NQ = 0, NO = 0, NE = 0;
  for (int r = 0; r < n_req; ++r) {
    const int P = n_tokens[r] + n_embeds[r];
    if (n_tokens[r] < 0 || n_embeds[r] < 0 || P < 1) return fail(S1_ERR_INVALID_ARG, "request %d: empty prefix", r);
    if (!valid_state(m, states[r])) return fail(S1_ERR_INVALID_HANDLE, "request %d: invalid state", r);
    if (P > states[r]->cap) return fail(S1_ERR_BUDGET, "request %d: prefix %d rows > state capacity %d", r, P, states[r]->cap);
    if (n_q[r] < 0 || (n_q[r] > 0 && !qs[r])) return fail(S1_ERR_INVALID_ARG, "request %d: bad question array", r);
    if (n_tokens[r] > 0 && (!tokens || !tokens[r])) return fail(S1_ERR_INVALID_ARG, "request %d: NULL tokens", r);
    if (n_embeds[r] > 0 && (!embeds || !embeds[r])) return fail(S1_ERR_INVALID_ARG, "request %d: NULL embeds", r);
    if (!device_ptrs && n_tokens[r] > 0) {
      int rc = validate_ids(tokens[r], n_tokens[r], m->sh.vocab, "token");
      if (rc) return rc;
    }
    Rp += P;
    NE += n_embeds[r];
    for (int j = 0; j < n_q[r]; ++j) {
      int rc = validate_question(m, qs[r][j], j, !device_ptrs);
      if (rc) return rc;
      if (P + qs[r][j].n_suffix > m->max_pos) return fail(S1_ERR_BUDGET, "position budget exceeded");
      Rs += qs[r][j].n_suffix;
      NO += qs[r][j].n_options;
      NQ += 1;
    }
    if (Rp + Rs > m->sh.max_rows) return fail(S1_ERR_BUDGET, "%d rows exceed max_rows %d", Rp + Rs, m->sh.max_rows);
  }
  if (NQ == 0) return fail(S1_ERR_INVALID_ARG, "no questions");
  int rc = ensure_scratch(m, Rp + Rs, NO);
  if (rc) return rc;
  Meta mt;
  mt.n_first = n_req;
  int row = 0, erow = 0;
  for (int r = 0; r < n_req; ++r) {
    const int P = n_tokens[r] + n_embeds[r];
    mt.ctxs.push_back(CtxDesc{states[r]->S, states[r]->KV, P, states[r]->cap, states[r]->conv});
    mt.seqs.push_back(SeqDesc{row, P, 0, -1, r, 0});
    mt.max_len = std::max(mt.max_len, P);
    for (int i = 0; i < P; ++i) mt.row_seq.push_back(r);
    for (int i = 0; i < n_embeds[r]; ++i) mt.row_src.push_back(-1 - (erow + i));
    for (int i = 0; i < n_tokens[r]; ++i) mt.row_src.push_back(device_ptrs ? 0 : tokens[r][i]);
    erow += n_embeds[r];
    row += P;
  }
  mt.opt_off.push_back(0);
  for (int r = 0; r < n_req; ++r)
    for (int j = 0; j < n_q[r]; ++j) {
      const s1_question& q = qs[r][j];
      const int sidx = (int)mt.seqs.size();
      mt.seqs.push_back(SeqDesc{row, q.n_suffix, n_tokens[r] + n_embeds[r], r, -1, 0});
      mt.max_len = std::max(mt.max_len, q.n_suffix);
      for (int i = 0; i < q.n_suffix; ++i) {
        mt.row_src.push_back(device_ptrs ? 0 : q.suffix[i]);
        mt.row_seq.push_back(sidx);
      }
      mt.q_row.push_back(row + q.n_suffix - 1);
      mt.q_type.push_back(q.type);
      for (int o = 0; o < q.n_options; ++o) mt.opt_ids.push_back(device_ptrs ? 0 : q.option_ids[o]);
      mt.opt_off.push_back(mt.opt_off.back() + q.n_options);
      mt.max_opts = std::max(mt.max_opts, q.n_options);
      row += q.n_suffix;
    }
  rc = upload_meta(m, mt, cap ? &cap->meta : nullptr);
  if (rc) return rc;
  rc = run_captured(m, cap, [&]() -> int {
    if (device_ptrs) {
      int rr = 0, opt = 0;
      for (int r = 0; r < n_req; ++r) {
        rr += n_embeds[r];
        if (n_tokens[r] > 0)
          CK(cudaMemcpyAsync(mt.d_row_src + rr, tokens[r], n_tokens[r] * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
        rr += n_tokens[r];
      }
      for (int r = 0; r < n_req; ++r)
        for (int j = 0; j < n_q[r]; ++j) {
          const s1_question& q = qs[r][j];
          CK(cudaMemcpyAsync(mt.d_row_src + rr, q.suffix, q.n_suffix * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
          CK(cudaMemcpyAsync(mt.d_opt_ids + opt, q.option_ids, q.n_options * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
          rr += q.n_suffix;
          opt += q.n_options;
        }
    }
    if (NE > 0) {
      const size_t rowb = (size_t)m->sh.d_model * 2;
      size_t eoff = 0;
      for (int r = 0; r < n_req; ++r) {
        if (n_embeds[r] == 0) continue;
        CK(cudaMemcpyAsync((char*)m->sc.xn + eoff, embeds[r], n_embeds[r] * rowb,
                           device_ptrs ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, m->stream));
        if (!device_ptrs) m->h2d_bytes += (long long)(n_embeds[r] * rowb);
        eoff += n_embeds[r] * rowb;
      }
    }
    return run_forward(m, mt, reinterpret_cast<const bf16*>(m->sc.xn), d_probs, d_stats, d_hidden, want_lm);
  });
  if (rc) return rc;
  for (int r = 0; r < n_req; ++r) states[r]->P = n_tokens[r] + n_embeds[r];
  *NQ_out = NQ;
  *NO_out = NO;
  return S1_OK;
}

int s1_prefill_decide_batch(s1_model* m, int32_t n_req, const int32_t* const* tokens, const int32_t* n_tokens,
                            const void* const* embeds, const int32_t* n_embeds, const s1_question* const* qs,
                            const int32_t* n_q, s1_result* const* out, float* const* last_hidden,
                            s1_state** states_out) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (n_req < 1 || !n_tokens || !qs || !n_q || !out) return fail(S1_ERR_INVALID_ARG, "bad batch arguments");
  for (int r = 0; r < n_req; ++r)
    if (n_q[r] > 0 && !out[r]) return fail(S1_ERR_INVALID_ARG, "request %d: NULL results", r);
  std::vector<int32_t> ne(n_req, 0);
  if (n_embeds) ne.assign(n_embeds, n_embeds + n_req);
  std::vector<s1_state*> sts(n_req, nullptr);
  auto cleanup = [&](int rc) {
    for (s1_state* x : sts) s1_state_destroy(x);
    return rc;
  };
  for (int r = 0; r < n_req; ++r) {
    const int P = n_tokens[r] + ne[r];
    if (P < 1) return cleanup(fail(S1_ERR_INVALID_ARG, "request %d: empty prefix", r));
    if (P > m->sh.max_rows) return cleanup(fail(S1_ERR_BUDGET, "request %d: prefix %d > max_rows", r, P));
    int rc = new_state(m, P, &sts[r]);
    if (rc) return cleanup(rc);
  }
  bool want_hidden = false;
  if (last_hidden)
    for (int r = 0; r < n_req; ++r) want_hidden |= (last_hidden[r] != nullptr);
  int NQ = 0, NO = 0;
  // output slots are sized after validation: count first
  int nq_tot = 0, no_tot = 0;
  for (int r = 0; r < n_req; ++r)
    for (int j = 0; j < n_q[r]; ++j) { nq_tot++; no_tot += std::max(0, qs[r][j].n_options); }
  int rc = S1_OK;
  {
    int rows = 0;
    for (int r = 0; r < n_req; ++r) {
      rows += n_tokens[r] + ne[r];
      for (int j = 0; j < n_q[r]; ++j) rows += std::max(0, qs[r][j].n_suffix);
    }
    if (rows > m->sh.max_rows) return cleanup(fail(S1_ERR_BUDGET, "%d rows exceed max_rows %d", rows, m->sh.max_rows));
    rc = ensure_scratch(m, std::max(rows, 1), no_tot);
    if (rc) return cleanup(rc);
  }
  float *probs, *stats, *hidden;
  output_slots(m, nq_tot, no_tot, &probs, &stats, &hidden);
  rc = fused_impl(m, n_req, tokens, n_tokens, embeds, ne.data(), sts.data(), qs, n_q, false, probs, stats,
                  want_hidden ? hidden : nullptr, &NQ, &NO, wants_lm(n_req, n_q, out));
  if (!rc) rc = fetch_results(m, n_req, qs, n_q, NQ, NO, want_hidden, out, last_hidden);
  if (rc) return cleanup(rc);
  for (int r = 0; r < n_req; ++r) {
    if (states_out) states_out[r] = sts[r];
    else s1_state_destroy(sts[r]);
  }
  return S1_OK;
}

int s1_prefill_decide(s1_model* m, const int32_t* tokens, int32_t n_tokens, const void* embeds, int32_t n_embeds,
                      const s1_question* qs, int32_t n_q, s1_result* out, float* last_hidden, s1_state** state_out) {
  const void* e[1] = {embeds};
  return s1_prefill_decide_batch(m, 1, &tokens, &n_tokens, e, &n_embeds, &qs, &n_q, &out, &last_hidden, state_out);
}

int s1_prefill_decide_async(s1_model* m, s1_state* st, const int32_t* d_tokens, int32_t n_tokens,
                            const void* d_embeds, int32_t n_embeds, const s1_question* qs_dev, int32_t n_q,
                            float* d_probs, float* d_stats, float* d_last_hidden) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (!valid_state(m, st)) return fail(S1_ERR_INVALID_HANDLE, "invalid state");
  if (!d_probs || !d_stats) return fail(S1_ERR_INVALID_ARG, "NULL output");
  const void* e[1] = {d_embeds};
  if (n_q < 1 || !qs_dev) return fail(S1_ERR_INVALID_ARG, "no questions");
  CallKey key('F');
  key.state(st, false).add(d_tokens).add(n_tokens).add(d_embeds).add(n_embeds);
  key.add(d_probs).add(d_stats).add(d_last_hidden).add(n_q);
  for (int j = 0; j < n_q; ++j) key.question(qs_dev[j]);
  return graph_call(
      m, key,
      [&](s1_model::Graph* cap) {
        int NQ = 0, NO = 0;
        return fused_impl(m, 1, &d_tokens, &n_tokens, e, &n_embeds, &st, &qs_dev, &n_q, true, d_probs, d_stats,
                          d_last_hidden, &NQ, &NO, false, cap);
      },
      [&]() { st->P = n_tokens + n_embeds; });
}

int s1_prefill_decide_batch_async(s1_model* m, int32_t n_req, s1_state* const* states,
                                  const int32_t* const* d_tokens, const int32_t* n_tokens,
                                  const void* const* d_embeds, const int32_t* n_embeds,
                                  const s1_question* const* qs_dev, const int32_t* n_q, float* d_probs,
                                  float* d_stats, float* d_last_hidden) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (n_req < 1 || !states || !d_tokens || !n_tokens || !qs_dev || !n_q)
    return fail(S1_ERR_INVALID_ARG, "bad batch arguments");
  if (!d_probs || !d_stats) return fail(S1_ERR_INVALID_ARG, "NULL output");
  std::vector<int32_t> ne(n_req, 0);
  std::vector<const void*> de(n_req, nullptr);
  if (n_embeds) ne.assign(n_embeds, n_embeds + n_req);
  if (d_embeds) de.assign(d_embeds, d_embeds + n_req);
  CallKey key('B');
  key.add(n_req).add(d_probs).add(d_stats).add(d_last_hidden);
  for (int r = 0; r < n_req; ++r) {
    if (!valid_state(m, states[r])) return fail(S1_ERR_INVALID_HANDLE, "request %d: invalid state", r);
    if (n_q[r] < 1 || !qs_dev[r]) return fail(S1_ERR_INVALID_ARG, "request %d: no questions", r);
    key.state(states[r], false).add(d_tokens[r]).add(n_tokens[r]).add(de[r]).add(ne[r]).add(n_q[r]);
    for (int j = 0; j < n_q[r]; ++j) key.question(qs_dev[r][j]);
  }
  return graph_call(
      m, key,
      [&](s1_model::Graph* cap) {
        int NQ = 0, NO = 0;
        return fused_impl(m, n_req, d_tokens, n_tokens, de.data(), ne.data(), states, qs_dev, n_q, true, d_probs,
                          d_stats, d_last_hidden, &NQ, &NO, false, cap);
      },
      [&]() {
        for (int r = 0; r < n_req; ++r) states[r]->P = n_tokens[r] + ne[r];
      });
}

int s1_set_graphs(s1_model* m, int enable) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  CK(cudaStreamSynchronize(m->stream));
  if (!enable) drop_graphs(m);
  m->graphs = enable != 0;
  return S1_OK;
}

// -- instrumentation ---------------------------------------------------------------------
int s1_profile(s1_model* m, int enable) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  CK(cudaStreamSynchronize(m->stream));
  if (enable && !m->prof) ++pdl_suppressed();
  if (!enable && m->prof) --pdl_suppressed();
  m->prof = enable != 0;
  m->prof_ev.clear();
  m->ev_next = 0;
  for (int c = 0; c < S1_PROF_NCLASS; ++c) {
    m->prof_flops[c] = m->prof_bytes[c] = 0;
    m->prof_count[c] = 0;
  }
  return S1_OK;
}

int s1_profile_read(s1_model* m, double* ms, double* flops, double* bytes, long* count) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  CK(cudaStreamSynchronize(m->stream));
  for (int c = 0; c < S1_PROF_NCLASS; ++c) {
    if (ms) ms[c] = 0;
    if (flops) flops[c] = m->prof_flops[c];
    if (bytes) bytes[c] = m->prof_bytes[c];
    if (count) count[c] = m->prof_count[c];
  }
  for (auto& pe : m->prof_ev) {
    float t = 0;
    CK(cudaEventElapsedTime(&t, pe.second.first, pe.second.second));
    if (ms) ms[pe.first] += t;
  }
  return S1_OK;
}

int s1_counters(s1_model* m, long long* launches, long long* h2d_bytes, long long* d2h_bytes) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  if (launches) *launches = m->launches;
  if (h2d_bytes) *h2d_bytes = m->h2d_bytes;
  if (d2h_bytes) *d2h_bytes = m->d2h_bytes;
  return S1_OK;
}

int s1_set_layer_trace(s1_model* m, float* d_trace, long long capacity_floats) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  AllocScope alloc_scope(m);
  if (d_trace && capacity_floats <= 0) return fail(S1_ERR_INVALID_ARG, "layer trace needs a positive capacity");
  CK(cudaStreamSynchronize(m->stream));
  m->trace = d_trace;
  m->trace_floats = d_trace ? capacity_floats : 0;
  return S1_OK;
}

int s1_set_gemm_impl(s1_model* m, int impl) {
  if (!valid_model(m)) return fail(S1_ERR_INVALID_HANDLE, "invalid model");
  if (impl != 0 && impl != 1) return fail(S1_ERR_INVALID_ARG, "impl must be 0 (tensor cores) or 1 (SIMT)");
  m->gemm_impl = impl;
  return S1_OK;
}

}  // extern "C"
