// Model runtime: weights, shared paged KV cache, workspace, the streamed
// originals of offloaded layers, the decoder forward, and the SubSpec decode
// loop (draft D levels -> verify the tree in one target pass -> accept ->
// compact), optionally captured once as a CUDA graph and replayed per cycle.
//
// Method: "SubSpec: Using the Target Model's Own Low-Bit Shadow as Its Draft
// Model" (2.1 offloading, 2.2 Step 4 substitutes + sharing + prefetch, 6.3
// tree verification) and "Speculate Deep and Accurate" (card: Approach and the
// measured effects of shared KV, sharpening and asynchronous transfer).
//
// Streams: the compute stream runs every kernel; a copy stream moves the bf16
// originals of offloaded layers from pinned host memory into a device ring of
// staging slots.  A target pass waits per layer for its slot to be staged;
// the copies for the first ring-full of layers are issued at the start of a
// cycle, so they run under the draft.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <mutex>
#include <vector>
#include "attn.cuh"
#include "gemm.cuh"
#include "layers.cuh"
#include "tree.cuh"

namespace sub {

struct Matrices {
  const void* w[7];   // wq wk wv wo wg wu wd (bf16 or packed codes)
  const uint16_t* s[7];
  const uint16_t* z[7];
  int bits[7];        // code bits of the substitutes (0 for bf16)
};

// Decode state on the device (one int each).
enum {
  ST_N = 0, ST_EMITTED = 1, ST_NACC = 2, ST_BONUS = 3, ST_TIES = 4,
  ST_DLIM = 5,     // adaptive depth: levels drafted this cycle
  ST_CONT = 6,     // adaptive depth: 1 while drafting goes on
  ST_LEVELS = 7,   // adaptive depth: levels drafted since the prefill
  ST_COUNT = 8
};

// Emitted tokens whose top-2 choice scores differ by less than this are
// counted as near-ties (sub_stats.near_tie_events).
constexpr float NEAR_TIE_GAP = 1e-2f;

}  // namespace sub

struct sub_model {
  sub_model_desc d{};
  std::vector<sub_layer_desc> layers;
  int qkv_dim = 0, q_dim = 0, kv_dim = 0;
  int rows_max = 0;         // largest forward (tree or prompt)
  int logit_rows = 0;
  int64_t dev_bytes = 0;
  std::vector<void*> allocs;
  // cache
  uint16_t* kpool = nullptr;
  uint16_t* vpool = nullptr;
  int32_t* page_table = nullptr;
  int page_size = 64, n_pages = 0;
  int64_t capacity = 0;
  float2* rope = nullptr;
  int max_pos = 0;
  // activations
  float* x = nullptr;        // [rows, H]
  float* xsave = nullptr;    // [tree slots, H]: residual stream at layer n_resident (verify reuse)
  // draft attention over long key ranges (32 key splits): cross-cluster
  // partials and counters, sized for the draft's widest level
  float* attn_x = nullptr;
  size_t attn_x_floats = 0;
  unsigned int* attn_xcnt = nullptr;
  uint16_t* xn = nullptr;    // [rows, H]
  float* qkv = nullptr;      // [rows, qkv_dim]
  uint16_t* q = nullptr;     // [rows, Hq*D]
  uint16_t* attn = nullptr;  // [rows, Hq*D]
  uint16_t* act = nullptr;   // [rows, F]
  float* logits = nullptr;   // [logit_rows, V]
  int32_t* rows_tok = nullptr;  // [rows] token ids staged for a forward
  float* split_part = nullptr;       // GEMV split-K partial sums
  size_t split_cap = 0;
  unsigned int* split_cnt = nullptr;
  int split_cnt_cap = 0;
  float* norm_partial = nullptr;     // [2][norm_parts] per-tile sums of squares of the
                                     // factored RMSNorms' inputs: attention, FFN
  int norm_parts = 0;
  // tree + decode state
  sub_tree tree{};
  int32_t* state = nullptr;
  int32_t* accepted = nullptr;
  int32_t* choice = nullptr;
  int32_t* out_tokens = nullptr;
  int out_cap = 0;
  int32_t* hist = nullptr;
  unsigned long long* part_key = nullptr;
  unsigned long long* part_key2 = nullptr;   // accept: runner-up keys (near-ties)
  float* part_f = nullptr;
  unsigned int* counters = nullptr;   // [0] expand, [1] accept
  size_t part_keys = 0, part_floats = 0;
  // staging ring
  int n_off = 0, ring = 0;
  size_t layer_bytes = 0;
  size_t mat_off[7] = {};
  size_t mat_bytes[7] = {};
  std::vector<uint16_t*> slots;
  cudaStream_t s_main = nullptr, s_copy = nullptr;
  cudaStream_t s_cond = nullptr;   // captures the bodies of conditional draft levels
  int64_t cond_kernels = 0;         // kernel nodes inside them (last capture)
  std::vector<cudaEvent_t> ev_staged, ev_free;
  // timing (recorded as graph event nodes inside a captured cycle): cycle
  // start, draft end, verify end; per offloaded layer, the compute stream
  // reaching it in a target pass and its copy finishing
  cudaEvent_t ev_cyc[3] = {};
  std::vector<cudaEvent_t> ev_ready, ev_tstaged;
  unsigned int timeouts0 = 0;   // pipeline timeouts seen at the last prefill
  int alloc_index = 0;          // device allocations made (fault injection)
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_t0 = nullptr, ev_t1 = nullptr;
  int32_t* host_state = nullptr;   // pinned
  int32_t* host_prompt = nullptr;  // pinned [max_prompt]
  int32_t* host_out = nullptr;     // pinned [out_cap]
  cudaEvent_t ev_g0 = nullptr, ev_g1 = nullptr, ev_g2 = nullptr;
  int n_prompt = 0;
  int64_t cycles = 0;
  int64_t max_emit = 0;
  int64_t graph_kernels = 0;
  // optional per-kernel tracing of eager forwards (SUB_TRACE=<file>)
  std::vector<std::pair<const char*, cudaEvent_t>> trace;
  std::vector<cudaEvent_t> trace_pool;
  size_t trace_used = 0;
  // graph of one decode cycle
  cudaGraphExec_t graph = nullptr;
  sub_decode_cfg graph_cfg{};
};

namespace sub {

static int32_t dalloc(sub_model* m, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  if (fault_injected("alloc", m->alloc_index++)) {
    *p = nullptr;
    return fail(SUB_ENOMEM, "cudaMalloc(" + std::to_string(bytes) + "): injected fault (SUB_FAULT)");
  }
  const cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    return fail(SUB_ENOMEM, std::string("cudaMalloc(") + std::to_string(bytes) +
                                "): " + cudaGetErrorString(e));
  }
  m->allocs.push_back(*p);
  m->dev_bytes += (int64_t)bytes;
  return SUB_OK;
}
template <class T>
static int32_t dalloc_t(sub_model* m, T** p, size_t count) {
  return dalloc(m, reinterpret_cast<void**>(p), count * sizeof(T));
}

static void free_model(sub_model* m) {
  if (!m) return;
  if (m->s_main) cudaStreamSynchronize(m->s_main);
  if (m->s_copy) cudaStreamSynchronize(m->s_copy);
  if (m->graph) cudaGraphExecDestroy(m->graph);
  for (void* p : m->allocs) cudaFree(p);
  for (cudaEvent_t e : m->trace_pool) cudaEventDestroy(e);
  for (cudaEvent_t e : m->ev_staged) cudaEventDestroy(e);
  for (cudaEvent_t e : m->ev_free) cudaEventDestroy(e);
  for (cudaEvent_t e : m->ev_ready) cudaEventDestroy(e);
  for (cudaEvent_t e : m->ev_tstaged) cudaEventDestroy(e);
  for (cudaEvent_t e : m->ev_cyc)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : {m->ev_fork, m->ev_join, m->ev_t0, m->ev_t1})
    if (e) cudaEventDestroy(e);
  if (m->s_main) cudaStreamDestroy(m->s_main);
  if (m->s_copy) cudaStreamDestroy(m->s_copy);
  if (m->s_cond) cudaStreamDestroy(m->s_cond);
  if (m->host_state) cudaFreeHost(m->host_state);
  if (m->host_prompt) cudaFreeHost(m->host_prompt);
  if (m->host_out) cudaFreeHost(m->host_out);
  for (cudaEvent_t e : {m->ev_g0, m->ev_g1, m->ev_g2})
    if (e) cudaEventDestroy(e);
  delete m;
}

static const uint16_t* const* mats_of(const sub_layer_desc& L) {
  static thread_local const uint16_t* p[7];
  p[0] = L.wq; p[1] = L.wk; p[2] = L.wv; p[3] = L.wo; p[4] = L.wg; p[5] = L.wu; p[6] = L.wd;
  return p;
}

// Weights of layer l for the target (staged originals when offloaded) or the draft.
static Matrices layer_mats(const sub_model* m, int l, bool draft) {
  Matrices r{};
  const sub_layer_desc& L = m->layers[l];
  const bool off = l >= m->d.n_resident;
  if (off && draft) {
    const sub_w4* w4[7] = {&L.q4, &L.k4, &L.v4, &L.o4, &L.g4, &L.u4, &L.d4};
    for (int i = 0; i < 7; ++i) {
      r.w[i] = w4[i]->q;
      r.s[i] = w4[i]->scale;
      r.z[i] = w4[i]->zero;
      r.bits[i] = w4[i]->bits ? w4[i]->bits : 4;
    }
  } else if (off) {
    const uint8_t* base = reinterpret_cast<const uint8_t*>(m->slots[(l - m->d.n_resident) % m->ring]);
    for (int i = 0; i < 7; ++i) r.w[i] = base + m->mat_off[i];
  } else {
    const uint16_t* const* p = mats_of(L);
    for (int i = 0; i < 7; ++i) r.w[i] = p[i];
  }
  return r;
}

// ---------------------------------------------------------------- streaming --
// Timing marks go in as event nodes when a cycle is captured (an ordinary
// record otherwise), so that each replay records them.
static cudaError_t mark(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t q = cudaStreamIsCapturing(st, &cs);
  if (q != cudaSuccess) return q;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(e, st, cudaEventRecordExternal)
             : cudaEventRecord(e, st);
}

static int32_t issue_copy(sub_model* m, int j) {
  if (fault_injected("h2d", j))
    return fail(SUB_ECUDA, "cudaMemcpyAsync (offloaded layer " + std::to_string(j) +
                               "): injected fault (SUB_FAULT)");
  const sub_layer_desc& L = m->layers[m->d.n_resident + j];
  uint8_t* dst = reinterpret_cast<uint8_t*>(m->slots[j % m->ring]);
  const uint16_t* const* src = mats_of(L);
  for (int i = 0; i < 7; ++i)
    SUB_CUDA_TRY(cudaMemcpyAsync(dst + m->mat_off[i], src[i], m->mat_bytes[i],
                                 cudaMemcpyHostToDevice, m->s_copy));
  SUB_CUDA_TRY(cudaEventRecord(m->ev_staged[j], m->s_copy));
  SUB_CUDA_TRY(mark(m->ev_tstaged[j], m->s_copy));
  return SUB_OK;
}

// Fork the copy stream off the compute stream and stage the first ring-full.
static int32_t begin_target_pass(sub_model* m) {
  if (m->n_off == 0) return SUB_OK;
  SUB_CUDA_TRY(cudaEventRecord(m->ev_fork, m->s_main));
  SUB_CUDA_TRY(cudaStreamWaitEvent(m->s_copy, m->ev_fork, 0));
  for (int j = 0; j < std::min(m->ring, m->n_off); ++j) SUB_TRY(issue_copy(m, j));
  return SUB_OK;
}
// Join the copy stream back (always, so a capture ends with both streams joined).
static int32_t end_target_pass(sub_model* m) {
  if (m->n_off == 0) return SUB_OK;
  SUB_CUDA_TRY(cudaEventRecord(m->ev_join, m->s_copy));
  SUB_CUDA_TRY(cudaStreamWaitEvent(m->s_main, m->ev_join, 0));
  return SUB_OK;
}

// ------------------------------------------------------------------ tracing --
// With SUB_TRACE=<file>, eager forwards record an event before every kernel on
// the compute stream; sub_model_forward then appends "name,ms" lines (kernel
// plus launch gap, stream order) to the file.  Off inside graph capture.
static const char* trace_path() {
  static const char* p = getenv("SUB_TRACE");
  return (p && p[0]) ? p : nullptr;
}
static void trace_mark(sub_model* m, const char* name) {
  if (!trace_path()) return;
  cudaStreamCaptureStatus cs;
  if (cudaStreamIsCapturing(m->s_main, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
  if (m->trace_used == m->trace_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return;
    m->trace_pool.push_back(e);
  }
  cudaEvent_t e = m->trace_pool[m->trace_used++];
  cudaEventRecord(e, m->s_main);
  m->trace.emplace_back(name, e);
}
static void trace_flush(sub_model* m) {
  if (!trace_path() || m->trace.size() < 2) {
    m->trace.clear();
    m->trace_used = 0;
    return;
  }
  cudaStreamSynchronize(m->s_main);
  FILE* f = fopen(trace_path(), "a");
  for (size_t i = 0; i + 1 < m->trace.size(); ++i) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, m->trace[i].second, m->trace[i + 1].second);
    if (f) fprintf(f, "%s,%.5f\n", m->trace[i].first, ms);
  }
  if (f) fclose(f);
  m->trace.clear();
  m->trace_used = 0;
}

// ------------------------------------------------------------------ forward --
struct FwdRows {
  const int32_t* tokens;   // [n]
  int n;
  int slot0;
  const int32_t* depth;    // [n] or null (chain)
  const int32_t* anc;      // [n, stride] or null (chain)
  int anc_stride;
  int n_slots;
  int64_t base;            // committed length (host) ...
  const int32_t* base_dev; // ... or on the device
  int64_t keys_hint;       // for the split heuristic
  // layer range [layer0, layer_end) (layer_end 0: all layers, then the head);
  // x_in / x_out: per-slot residual streams [slots, hidden] fp32 to start
  // from (instead of the embedding) and to leave at layer_end
  int layer0;
  int layer_end;
  const float* x_in;
  float* x_out;
};

static GemvArgs mm_args(const void* X, int M, int K, const Matrices& W, const int* idx, int nseg,
                        const int* rows, void* Y, int ldy, const sub_model* m = nullptr) {
  GemvArgs a{};
  if (m) {
    a.split_part = m->split_part;
    a.split_cap = m->split_cap;
    a.split_cnt = m->split_cnt;
    a.split_cnt_cap = m->split_cnt_cap;
  }
  a.X = reinterpret_cast<const uint16_t*>(X);
  a.M = M;
  a.K = K;
  a.ldx = K;
  int acc = 0;
  for (int i = 0; i < nseg; ++i) {
    a.W[i] = W.w[idx[i]];
    a.S[i] = W.s[idx[i]];
    a.Z[i] = W.z[idx[i]];
    acc += rows[i];
    a.seg_end[i] = acc;
  }
  a.n_seg = nseg;
  a.N = acc;
  a.Y = Y;
  a.ldy = ldy;
  a.bits = W.bits[idx[0]];   // segments of one launch share their width (checked at create)
  return a;
}

static int32_t forward(sub_model* m, bool draft, const FwdRows& r, float* logits, bool last_only) {
  const sub_model_desc& d = m->d;
  const cudaStream_t st = m->s_main;
  const int H = d.hidden, F = d.ffn, D = d.head_dim;
  const int M = r.n;
  // Draft-shaped passes (M <= 16) run the GEMV kernels with fused epilogues:
  // RoPE + KV store after q/k/v, the next RMSNorm after each residual add.
  // Tree-shaped passes run the tiled GEMM with separate row kernels.
  const bool fused = M <= 16;
  // SUB_FUSE_NORM=0 runs the RMSNorms as their own kernels on this path too
  static const bool fuse_norm_env = env_flag("SUB_FUSE_NORM", true);
  static const bool fuse_qkv_env = env_flag("SUB_FUSE_QKV", true);
  const bool fuse_norm = fused && fuse_norm_env;
  const bool fuse_qkv = fused && fuse_qkv_env;
  RowSet rs{};
  rs.tokens = r.tokens;
  rs.depth = r.depth;
  rs.slot0 = r.slot0;
  rs.base = r.base;
  rs.base_dev = r.base_dev;
  trace_mark(m, "embed");
  // Fused path: RMSNorm in factored form.  xn holds bf16(x * gain), the
  // producer leaves per-tile sums of squares, and the consumer GEMV scales its
  // sums by the row's rsqrt(mean(x^2) + eps), formed from those parts.
  const int tiles = (H + 15) / 16;
  RowScale r_attn{}, r_ffn{};
  if (fuse_norm) {
    r_attn = RowScale{m->norm_partial, 1, H, d.rms_eps, 0};   // the embedding: one part
    r_ffn = RowScale{m->norm_partial + m->norm_parts, tiles, H, d.rms_eps, 0};
  }
  const int l0 = r.layer0, l1 = r.layer_end ? r.layer_end : d.n_layers;
  if (r.x_in)
    SUB_TRY(launch_rows_in(r.x_in + (size_t)r.slot0 * H, H, M, m->x, m->layers[l0].attn_norm,
                           d.rms_eps, m->xn, fuse_norm ? m->norm_partial : nullptr, st));
  else
    SUB_TRY(launch_embed(d.embed, H, rs, M, m->x, m->layers[0].attn_norm, d.rms_eps, m->xn,
                         fuse_norm ? m->norm_partial : nullptr, st));

  AttnArgs at{};
  at.Q = m->q;
  at.O = m->attn;
  at.n_q = M;
  at.n_heads_q = d.n_heads_q;
  at.n_heads_kv = d.n_heads_kv;
  at.head_dim = D;
  at.k = m->kpool;
  at.v = m->vpool;
  at.page_table = m->page_table;
  at.page_size = m->page_size;
  at.n_pages = m->n_pages;
  at.n_prefix = r.base;
  at.n_prefix_dev = r.base_dev;
  at.tree_base = r.base;
  at.tree_base_dev = r.base_dev;
  at.n_slots = r.n_slots;
  at.anc = r.anc;
  at.anc_stride = r.anc_stride;
  at.depth = r.depth;
  at.chain_slot0 = r.slot0;
  at.scale = 1.0f / sqrtf((float)D);
  at.early_reads = 1;   // predecessors signal only after their own wait
  const bool two_level = m->attn_x && attn_xpart_floats(at, 32) <= m->attn_x_floats;
  const int splits = attn_pick_splits(at, (int)std::min<int64_t>(r.keys_hint, 1 << 30), two_level);
  if (splits > ATTN_MAX_SPLIT) {
    const size_t rows = attn_xpart_floats(at, splits) / (D + 2);
    at.xpart = m->attn_x;
    at.xm = m->attn_x + rows * D;
    at.xl = at.xm + rows;
    at.xcnt = m->attn_xcnt;
  }

  QkvPostArgs qp{};
  qp.qkv = m->qkv;
  qp.rows = M;
  qp.n_heads_q = d.n_heads_q;
  qp.n_heads_kv = d.n_heads_kv;
  qp.head_dim = D;
  qp.rope = m->rope;
  qp.max_pos = m->max_pos;
  qp.rs = rs;
  qp.q_out = m->q;
  qp.k_cache = m->kpool;
  qp.v_cache = m->vpool;
  qp.page_table = m->page_table;
  qp.page_size = m->page_size;
  qp.n_pages = m->n_pages;

  QkvOut qo{};
  qo.n_heads_q = d.n_heads_q;
  qo.n_heads_kv = d.n_heads_kv;
  qo.head_dim = D;
  qo.rope = m->rope;
  qo.max_pos = m->max_pos;
  qo.depth = r.depth;
  qo.slot0 = r.slot0;
  qo.base = r.base;
  qo.base_dev = r.base_dev;
  qo.q_out = m->q;
  qo.k_cache = m->kpool;
  qo.v_cache = m->vpool;
  qo.page_table = m->page_table;
  qo.page_size = m->page_size;
  qo.n_pages = m->n_pages;

  auto norm_out = [&](const uint16_t* gain, const RowScale& to) {
    NormOut no{};
    no.xn = m->xn;
    no.gain = gain;
    no.partial = const_cast<float*>(to.partial);
    return no;
  };

  const int qkv_rows[3] = {m->q_dim, m->kv_dim, m->kv_dim};
  const int qkv_idx[3] = {0, 1, 2};
  const int o_rows[1] = {H};
  const int o_idx[1] = {3};
  const int gu_rows[2] = {F, F};
  const int gu_idx[2] = {4, 5};
  const int dn_idx[1] = {6};

  for (int l = l0; l < l1; ++l) {
    const sub_layer_desc& L = m->layers[l];
    const bool off = l >= d.n_resident;
    const bool w4 = off && draft;
    const int j = l - d.n_resident;
    if (off && !draft) {
      SUB_CUDA_TRY(mark(m->ev_ready[j], st));
      SUB_CUDA_TRY(cudaStreamWaitEvent(st, m->ev_staged[j], 0));
    }
    const Matrices W = layer_mats(m, l, draft);
    const uint16_t* next_gain = l + 1 < d.n_layers ? m->layers[l + 1].attn_norm : d.final_norm;

    trace_mark(m, w4 ? "qkv_w4" : "qkv_bf16");
    if (fuse_qkv) {
      if (!fuse_norm && l > l0) SUB_TRY(launch_rmsnorm(m->x, L.attn_norm, M, H, d.rms_eps, m->xn, st));
      GemvArgs qa = mm_args(m->xn, M, H, W, qkv_idx, 3, qkv_rows, nullptr, 0, m);
      qa.xscale = r_attn;
      qo.layer = l;
      qa.qkv = qo;
      SUB_TRY(launch_gemv(qa, w4, EPI_QKV, st));
    } else {
      if (l > l0 && !fuse_norm) SUB_TRY(launch_rmsnorm(m->x, L.attn_norm, M, H, d.rms_eps, m->xn, st));
      GemvArgs qa = mm_args(m->xn, M, H, W, qkv_idx, 3, qkv_rows, m->qkv, m->qkv_dim, m);
      qa.xscale = r_attn;
      SUB_TRY(launch_matmul(qa, w4, EPI_F32, st));
      qp.layer = l;
      SUB_TRY(launch_qkv_post(qp, st));
    }
    at.layer = l;
    trace_mark(m, "attn");
    SUB_TRY(launch_tree_attn(at, splits, st));
    trace_mark(m, w4 ? "o_w4" : "o_bf16");
    {
      GemvArgs oa = mm_args(m->attn, M, m->q_dim, W, o_idx, 1, o_rows, m->x, H, m);
      if (fuse_norm) {
        oa.norm = norm_out(L.ffn_norm, r_ffn);
        SUB_TRY(launch_gemv(oa, w4, EPI_RESID, st));
      } else {
        SUB_TRY(launch_matmul(oa, w4, EPI_RESID, st));
        SUB_TRY(launch_rmsnorm(m->x, L.ffn_norm, M, H, d.rms_eps, m->xn, st));
      }
    }
    trace_mark(m, w4 ? "gate_up_w4" : "gate_up_bf16");
    {
      GemvArgs ga = mm_args(m->xn, M, H, W, gu_idx, 2, gu_rows, m->act, F, m);
      ga.N = F;   // GLU: grid covers one segment's rows
      ga.xscale = r_ffn;
      SUB_TRY(launch_matmul(ga, w4, EPI_GLU, st));
    }
    trace_mark(m, w4 ? "down_w4" : "down_bf16");
    {
      GemvArgs da = mm_args(m->act, M, F, W, dn_idx, 1, o_rows, m->x, H, m);
      if (fuse_norm) {
        da.norm = norm_out(next_gain, r_attn);
        SUB_TRY(launch_gemv(da, w4, EPI_RESID, st));
        r_attn.n_parts = tiles;   // from here on the attention input comes from this GEMV
      } else {
        SUB_TRY(launch_matmul(da, w4, EPI_RESID, st));
      }
    }

    if (off && !draft) {
      // slot j % ring is free once this layer's kernels are done: stage layer j + ring
      if (j + m->ring < m->n_off) {
        SUB_CUDA_TRY(cudaEventRecord(m->ev_free[j], st));
        SUB_CUDA_TRY(cudaStreamWaitEvent(m->s_copy, m->ev_free[j], 0));
        SUB_TRY(issue_copy(m, j + m->ring));
      }
    }
  }
  if (r.x_out) SUB_TRY(launch_rows_out(m->x, H, M, r.x_out + (size_t)r.slot0 * H, st));
  if (l1 < d.n_layers) return SUB_OK;   // a leading part: no head
  // final norm (already in xn on the fused path) + lm_head
  const int first = last_only ? M - 1 : 0;
  const int nrow = last_only ? 1 : M;
  const uint16_t* xin = m->xn;
  if (fuse_norm) {
    xin = m->xn + (size_t)first * H;
  } else {
    SUB_TRY(launch_rmsnorm(m->x + (size_t)first * H, d.final_norm, nrow, H, d.rms_eps, m->xn, st));
  }
  trace_mark(m, "lm_head");
  if (logits) {
    Matrices lm{};
    lm.w[0] = d.lm_head;
    const int idx0[1] = {0};
    const int vrows[1] = {d.vocab};
    GemvArgs la = mm_args(xin, nrow, H, lm, idx0, 1, vrows, logits, d.vocab, m);
    la.xscale = r_attn;
    la.xscale.tok0 = first;
    SUB_TRY(launch_matmul(la, false, EPI_F32, st));
  }
  trace_mark(m, "end");
  return SUB_OK;
}

// ------------------------------------------------------------ tiny kernels --
// Kernel nodes at the top level of a graph.
static int64_t count_kernels(cudaGraph_t g) {
  size_t n = 0;
  if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess || n == 0) return 0;
  std::vector<cudaGraphNode_t> nodes(n);
  if (cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return 0;
  int64_t k = 0;
  for (auto nd : nodes) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nd, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++k;
  }
  return k;
}

// Adaptive depth, after the expansion of level `level`: the new nodes (depth
// level + 1) are slots s0 .. s0 + k - 1.  Drafting goes on -- the next level's
// conditional node runs -- when their best cumulative score is >= stop.
__global__ void adapt_kernel(const float* score, int s0, int k, float stop, int32_t* state,
                             int level, cudaGraphConditionalHandle next, int has_next) {
  pdl_wait();
  pdl_trigger();
  float mx = -INFINITY;
  for (int i = threadIdx.x; i < k; i += 32) mx = fmaxf(mx, score[s0 + i]);
  mx = warp_max(mx);
  if (threadIdx.x == 0) {
    const unsigned go = mx >= stop ? 1u : 0u;
    state[ST_DLIM] = level + 1;
    state[ST_CONT] = (int)go;
    state[ST_LEVELS] += 1;
    if (has_next) cudaGraphSetConditional(next, go);
  }
}

// After accept: committed length += accepted + 1, the bonus becomes the root.
__global__ void advance_kernel(int32_t* state, int32_t* root_token) {
  pdl_wait();
  pdl_trigger();
  state[ST_N] += state[ST_NACC] + 1;
  *root_token = state[ST_BONUS];
}

}  // namespace sub

using namespace sub;

// ------------------------------------------------------------------ create --
extern "C" int32_t sub_model_create(const sub_model_desc* desc, sub_model** out) {
  SUB_CHECK_ARG(desc && out && desc->layers, "null pointer");
  const sub_model_desc& d = *desc;
  SUB_CHECK_ARG(d.n_layers >= 1 && d.hidden >= 64 && d.hidden % 64 == 0, "bad n_layers/hidden");
  SUB_CHECK_ARG(d.head_dim == 64 || d.head_dim == 128, "head_dim must be 64 or 128");
  SUB_CHECK_ARG(d.n_heads_kv >= 1 && d.n_heads_q % d.n_heads_kv == 0, "Hq % Hkv != 0");
  SUB_CHECK_ARG(d.ffn % 16 == 0 && d.vocab >= 16 && d.vocab <= (1 << 20), "bad ffn/vocab");
  SUB_CHECK_ARG(d.n_resident >= 0 && d.n_resident <= d.n_layers, "bad n_resident");
  SUB_CHECK_ARG(d.max_seq >= 2 && d.max_prompt >= 1 && d.max_prompt <= d.max_seq, "bad max_seq");
  SUB_CHECK_ARG(d.max_depth >= 0 && d.max_depth <= 64 && d.max_width >= 1 &&
                    d.max_width <= MAX_WIDTH,
                "tree size out of range (depth <= 64, width <= 16)");
  SUB_CHECK_ARG(d.embed && d.lm_head && d.final_norm, "null global weights");
  *out = nullptr;
  sub_model* m = new sub_model();
  m->d = d;
  m->layers.assign(d.layers, d.layers + d.n_layers);
  m->d.layers = m->layers.data();
  auto bail = [&](int32_t code) {
    const std::string msg = sub_last_error();
    free_model(m);
    set_error(msg);
    return code;
  };
#define CREATE_TRY(expr) do { int32_t _s = (expr); if (_s != SUB_OK) return bail(_s); } while (0)
#define CREATE_CUDA(expr) do { cudaError_t _e = (expr); if (_e != cudaSuccess) { \
    fail(SUB_ECUDA, std::string(#expr) + ": " + cudaGetErrorString(_e)); return bail(SUB_ECUDA); } } while (0)

  for (int l = 0; l < d.n_layers; ++l) {
    const sub_layer_desc& L = d.layers[l];
    if (!(L.wq && L.wk && L.wv && L.wo && L.wg && L.wu && L.wd && L.attn_norm && L.ffn_norm)) {
      fail(SUB_EINVAL, "layer " + std::to_string(l) + ": null weight");
      return bail(SUB_EINVAL);
    }
    if (l >= d.n_resident) {
      const sub_w4* w4[7] = {&L.q4, &L.k4, &L.v4, &L.o4, &L.g4, &L.u4, &L.d4};
      for (auto* w : w4) {
        if (!(w->q && w->scale && w->zero)) {
          fail(SUB_EINVAL, "layer " + std::to_string(l) + ": null int4 substitute");
          return bail(SUB_EINVAL);
        }
        if (!(w->bits == 0 || w->bits == 2 || w->bits == 3 || w->bits == 4)) {
          fail(SUB_EINVAL, "layer " + std::to_string(l) + ": substitute bits must be 2, 3 or 4");
          return bail(SUB_EINVAL);
        }
      }
      auto b = [](const sub_w4& w) { return w.bits ? w.bits : 4; };
      if (b(L.q4) != b(L.k4) || b(L.q4) != b(L.v4) || b(L.g4) != b(L.u4)) {
        fail(SUB_EINVAL, "layer " + std::to_string(l) +
                             ": q/k/v substitutes must share one width, and so must gate/up");
        return bail(SUB_EINVAL);
      }
    }
  }
  CREATE_TRY(gemm_init());
  CREATE_TRY(gemv_init());
  CREATE_TRY(gemm_tc_init());
  CREATE_TRY(attn_init());
  CREATE_CUDA(cudaStreamCreateWithFlags(&m->s_main, cudaStreamNonBlocking));
  CREATE_CUDA(cudaStreamCreateWithFlags(&m->s_copy, cudaStreamNonBlocking));
  CREATE_CUDA(cudaStreamCreateWithFlags(&m->s_cond, cudaStreamNonBlocking));
  for (cudaEvent_t* e : {&m->ev_fork, &m->ev_join})
    CREATE_CUDA(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
  CREATE_CUDA(cudaEventCreateWithFlags(&m->ev_t0, cudaEventDisableTiming));
  CREATE_CUDA(cudaEventCreateWithFlags(&m->ev_t1, cudaEventDisableTiming));
  CREATE_CUDA(cudaEventCreate(&m->ev_g0));
  CREATE_CUDA(cudaEventCreate(&m->ev_g1));
  CREATE_CUDA(cudaEventCreate(&m->ev_g2));
  for (cudaEvent_t& e : m->ev_cyc) CREATE_CUDA(cudaEventCreate(&e));
  CREATE_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&m->host_state), 64, cudaHostAllocDefault));

  const int H = d.hidden, D = d.head_dim, F = d.ffn;
  m->q_dim = d.n_heads_q * D;
  m->kv_dim = d.n_heads_kv * D;
  m->qkv_dim = m->q_dim + 2 * m->kv_dim;
  const int n_tree = 1 + d.max_depth * d.max_width;
  m->rows_max = std::max({n_tree, d.max_prompt, d.max_width});
  m->logit_rows = std::max(n_tree, d.max_width);

  // cache: committed tokens + one tree region + a page of slack
  m->capacity = (int64_t)d.max_seq + n_tree + m->page_size;
  m->n_pages = (int)cdiv(m->capacity, m->page_size);
  m->capacity = (int64_t)m->n_pages * m->page_size;
  const size_t kv_elems = (size_t)d.n_layers * m->n_pages * d.n_heads_kv * m->page_size * D;
  CREATE_TRY(dalloc_t(m, &m->kpool, kv_elems));
  CREATE_TRY(dalloc_t(m, &m->vpool, kv_elems));
  CREATE_CUDA(cudaMemset(m->kpool, 0, kv_elems * 2));
  CREATE_CUDA(cudaMemset(m->vpool, 0, kv_elems * 2));
  {
    std::vector<int32_t> pt(m->n_pages);
    for (int i = 0; i < m->n_pages; ++i) pt[i] = i;
    CREATE_TRY(dalloc_t(m, &m->page_table, pt.size()));
    CREATE_CUDA(cudaMemcpy(m->page_table, pt.data(), pt.size() * 4, cudaMemcpyHostToDevice));
  }
  // RoPE table in double, stored fp32: angle = pos * theta^(-2i/D)
  {
    m->max_pos = (int)m->capacity;
    std::vector<float2> tab((size_t)m->max_pos * (D / 2));
    for (int p = 0; p < m->max_pos; ++p)
      for (int i = 0; i < D / 2; ++i) {
        const double ang = (double)p * std::pow((double)d.rope_theta, -2.0 * i / D);
        tab[(size_t)p * (D / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    CREATE_TRY(dalloc_t(m, &m->rope, tab.size()));
    CREATE_CUDA(cudaMemcpy(m->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
  }
  const size_t R = m->rows_max;
  CREATE_TRY(dalloc_t(m, &m->x, R * H));
  if (d.n_resident > 0 && d.max_depth > 0) {
    const size_t n_tree = 1 + (size_t)d.max_depth * d.max_width;
    CREATE_TRY(dalloc_t(m, &m->xsave, n_tree * H));
    CREATE_CUDA(cudaMemset(m->xsave, 0, n_tree * H * 4));
  }
  {
    AttnArgs w{};   // the draft's widest level, for 32-split attention
    w.n_q = std::max(d.max_width, 1);
    w.n_heads_q = d.n_heads_q;
    w.n_heads_kv = d.n_heads_kv;
    w.head_dim = D;
    m->attn_x_floats = attn_xpart_floats(w, 2 * ATTN_MAX_SPLIT);
    const size_t nc = attn_xcnt_count(w, 2 * ATTN_MAX_SPLIT);
    CREATE_TRY(dalloc_t(m, &m->attn_x, m->attn_x_floats));
    CREATE_TRY(dalloc_t(m, &m->attn_xcnt, nc));
    CREATE_CUDA(cudaMemset(m->attn_xcnt, 0, nc * 4));
  }
  CREATE_TRY(dalloc_t(m, &m->xn, R * H));
  CREATE_TRY(dalloc_t(m, &m->qkv, R * m->qkv_dim));
  CREATE_TRY(dalloc_t(m, &m->q, R * m->q_dim));
  CREATE_TRY(dalloc_t(m, &m->attn, R * m->q_dim));
  CREATE_TRY(dalloc_t(m, &m->act, R * F));
  CREATE_TRY(dalloc_t(m, &m->logits, (size_t)m->logit_rows * d.vocab));
  CREATE_TRY(dalloc_t(m, &m->rows_tok, R));
  m->split_cap = (size_t)1 << 24;            // 64 MB of partial sums
  m->split_cnt_cap = 8192;
  CREATE_TRY(dalloc_t(m, &m->split_part, m->split_cap));
  CREATE_TRY(dalloc_t(m, &m->split_cnt, m->split_cnt_cap));
  CREATE_CUDA(cudaMemset(m->split_cnt, 0, m->split_cnt_cap * 4));
  m->norm_parts = (H / 16 + 1) * 16;
  CREATE_TRY(dalloc_t(m, &m->norm_partial, 2 * m->norm_parts));

  // tree (slot 0 = root: parent -1, depth 0, score 0, anc [0, -1...])
  {
    const int A = d.max_depth + 1;
    m->tree.width = d.max_width;
    m->tree.max_depth = d.max_depth;
    CREATE_TRY(dalloc_t(m, &m->tree.token, n_tree));
    CREATE_TRY(dalloc_t(m, &m->tree.parent, n_tree));
    CREATE_TRY(dalloc_t(m, &m->tree.depth, n_tree));
    CREATE_TRY(dalloc_t(m, &m->tree.score, n_tree));
    CREATE_TRY(dalloc_t(m, &m->tree.anc, (size_t)n_tree * A));
    std::vector<int32_t> anc((size_t)n_tree * A, -1), par(n_tree, -1), dep(n_tree, 0);
    anc[0] = 0;
    CREATE_CUDA(cudaMemcpy(m->tree.anc, anc.data(), anc.size() * 4, cudaMemcpyHostToDevice));
    CREATE_CUDA(cudaMemcpy(m->tree.parent, par.data(), par.size() * 4, cudaMemcpyHostToDevice));
    CREATE_CUDA(cudaMemcpy(m->tree.depth, dep.data(), dep.size() * 4, cudaMemcpyHostToDevice));
    CREATE_CUDA(cudaMemset(m->tree.score, 0, n_tree * 4));
    CREATE_CUDA(cudaMemset(m->tree.token, 0, n_tree * 4));
  }
  CREATE_TRY(dalloc_t(m, &m->state, ST_COUNT));
  CREATE_TRY(dalloc_t(m, &m->accepted, std::max(d.max_depth, 1)));
  CREATE_TRY(dalloc_t(m, &m->choice, n_tree));
  CREATE_TRY(dalloc_t(m, &m->hist, d.max_depth + 1));
  m->out_cap = d.max_seq + d.max_depth + 2;
  CREATE_TRY(dalloc_t(m, &m->out_tokens, m->out_cap));
  CREATE_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&m->host_prompt), (size_t)d.max_prompt * 4,
                            cudaHostAllocDefault));
  CREATE_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&m->host_out), (size_t)m->out_cap * 4,
                            cudaHostAllocDefault));
  {
    const int ec = expand_pick_chunks(d.max_width, d.vocab);
    const int ac = std::max(accept_pick_chunks(n_tree, d.vocab), accept_pick_chunks(1, d.vocab));
    m->part_keys = std::max((size_t)d.max_width * 64 * MAX_WIDTH, (size_t)n_tree * 64);
    (void)ec;
    (void)ac;
    m->part_floats = (size_t)d.max_width * 64 * 2;
    CREATE_TRY(dalloc_t(m, &m->part_key, m->part_keys));
    CREATE_TRY(dalloc_t(m, &m->part_key2, m->part_keys));
    CREATE_TRY(dalloc_t(m, &m->part_f, m->part_floats));
    CREATE_TRY(dalloc_t(m, &m->counters, 4));
    CREATE_CUDA(cudaMemset(m->counters, 0, 16));
  }

  // staging ring for the offloaded originals
  m->n_off = d.n_layers - d.n_resident;
  if (m->n_off > 0) {
    const size_t rows[7] = {(size_t)m->q_dim, (size_t)m->kv_dim, (size_t)m->kv_dim, (size_t)H,
                            (size_t)F, (size_t)F, (size_t)H};
    const size_t cols[7] = {(size_t)H, (size_t)H, (size_t)H, (size_t)m->q_dim,
                            (size_t)H, (size_t)H, (size_t)F};
    size_t off = 0;
    for (int i = 0; i < 7; ++i) {
      m->mat_off[i] = off;
      m->mat_bytes[i] = rows[i] * cols[i] * 2;
      off += (m->mat_bytes[i] + 255) / 256 * 256;
    }
    m->layer_bytes = off;
    m->ring = d.staging_layers <= 0 ? m->n_off : std::min(d.staging_layers, m->n_off);
    for (int i = 0; i < m->ring; ++i) {
      void* p = nullptr;
      CREATE_TRY(dalloc(m, &p, m->layer_bytes));
      m->slots.push_back(reinterpret_cast<uint16_t*>(p));
    }
    m->ev_staged.resize(m->n_off, nullptr);
    m->ev_free.resize(m->n_off, nullptr);
    m->ev_ready.resize(m->n_off, nullptr);
    m->ev_tstaged.resize(m->n_off, nullptr);
    for (int j = 0; j < m->n_off; ++j) {
      CREATE_CUDA(cudaEventCreateWithFlags(&m->ev_staged[j], cudaEventDisableTiming));
      CREATE_CUDA(cudaEventCreateWithFlags(&m->ev_free[j], cudaEventDisableTiming));
      CREATE_CUDA(cudaEventCreate(&m->ev_ready[j]));
      CREATE_CUDA(cudaEventCreate(&m->ev_tstaged[j]));
    }
  }
  CREATE_CUDA(cudaMemset(m->xn, 0, R * H * 2));
  CREATE_CUDA(cudaMemset(m->attn, 0, R * m->q_dim * 2));
  CREATE_CUDA(cudaMemset(m->act, 0, R * F * 2));
  CREATE_CUDA(cudaDeviceSynchronize());
  *out = m;
  return SUB_OK;
#undef CREATE_TRY
#undef CREATE_CUDA
}

extern "C" int32_t sub_model_destroy(sub_model* m) {
  free_model(m);
  return SUB_OK;
}

extern "C" int32_t sub_model_memory(const sub_model* m, int64_t* device_bytes) {
  SUB_CHECK_ARG(m && device_bytes, "null pointer");
  *device_bytes = m->dev_bytes;
  return SUB_OK;
}

extern "C" int32_t sub_model_kv(sub_model* m, sub_kv_cache* out) {
  SUB_CHECK_ARG(m && out, "null pointer");
  out->k = m->kpool;
  out->v = m->vpool;
  out->page_table = m->page_table;
  out->n_layers = m->d.n_layers;
  out->n_heads_kv = m->d.n_heads_kv;
  out->head_dim = m->d.head_dim;
  out->page_size = m->page_size;
  out->n_pages = m->n_pages;
  out->capacity = m->capacity;
  return SUB_OK;
}

// ------------------------------------------------------------ forward (API) --
extern "C" int32_t sub_model_forward(sub_model* m, int32_t which, const int32_t* tokens,
                                     int32_t n_rows, int32_t slot0, const int32_t* depth,
                                     const int32_t* anc, int32_t anc_stride, int64_t n_prefix,
                                     float* logits, void* stream) {
  SUB_CHECK_ARG(m && tokens, "null pointer");
  SUB_CHECK_ARG(which == 0 || which == 1, "which must be 0 (target) or 1 (draft)");
  SUB_CHECK_ARG(n_rows >= 1 && n_rows <= m->rows_max, "n_rows out of range");
  SUB_CHECK_ARG(slot0 >= 0 && n_prefix >= 0, "negative slot or prefix");
  SUB_CHECK_ARG(n_prefix + slot0 + n_rows <= m->capacity, "beyond the cache capacity");
  SUB_CHECK_ARG(!anc || (depth && anc_stride >= 1), "anc needs depth and anc_stride");
  SUB_CHECK_ARG(n_prefix + slot0 + n_rows <= m->max_pos, "positions beyond the RoPE table");
  const cudaStream_t user = as_stream(stream);
  // order after the caller's stream, run on the model's streams, order back
  SUB_CUDA_TRY(cudaEventRecord(m->ev_t0, user));
  SUB_CUDA_TRY(cudaStreamWaitEvent(m->s_main, m->ev_t0, 0));
  FwdRows r{};
  r.tokens = tokens;
  r.n = n_rows;
  r.slot0 = slot0;
  r.depth = depth;
  r.anc = anc;
  r.anc_stride = anc_stride;
  r.n_slots = slot0 + n_rows;
  r.base = n_prefix;
  r.keys_hint = n_prefix + slot0 + n_rows;
  const bool target = which == 0;
  if (target) SUB_TRY(begin_target_pass(m));
  SUB_TRY(forward(m, !target, r, logits, false));
  if (target) SUB_TRY(end_target_pass(m));
  trace_flush(m);
  SUB_CUDA_TRY(cudaEventRecord(m->ev_t1, m->s_main));
  SUB_CUDA_TRY(cudaStreamWaitEvent(user, m->ev_t1, 0));
  return SUB_OK;
}

// ----------------------------------------------------------------- generate --
// Adaptive depth is on for a finite negative stop_logp (0, a zero-filled
// config, -inf and NaN all draft every level).
// Verify reuse needs resident layers to share and a tree.
static bool reuses(const sub_model* m, const sub_decode_cfg& c) {
  return c.verify_reuse && c.depth > 0 && m->d.n_resident > 0 && m->xsave;
}

static bool adaptive(const sub_decode_cfg& c) {
  return c.depth > 0 && c.stop_logp < 0.f && c.stop_logp > -INFINITY;
}

static int32_t accept_args(sub_model* m, const sub_decode_cfg& c, int n_nodes, AcceptArgs& a) {
  a = AcceptArgs{};
  a.logits = m->logits;
  a.V = m->d.vocab;
  a.tree = m->tree;
  a.tree.width = c.width;
  a.tree.max_depth = m->d.max_depth;
  a.n_nodes = n_nodes;
  a.mode = c.mode;
  a.temp = c.target_temp;
  a.seed = c.seed;
  a.root_pos_dev = m->state + ST_N;
  a.n_chunks = accept_pick_chunks(n_nodes, m->d.vocab);
  if ((size_t)n_nodes * a.n_chunks > m->part_keys) return fail(SUB_EINVAL, "accept scratch too small");
  a.part_key = m->part_key;
  a.counter = m->counters + 1;
  a.accepted = m->accepted;
  a.n_accepted = m->state + ST_NACC;
  a.bonus = m->state + ST_BONUS;
  a.choice = m->choice;
  a.out_tokens = m->out_tokens;
  a.state_emitted = m->state + ST_EMITTED;
  a.hist = m->hist;
  a.part_key2 = m->part_key2;
  a.near_ties = m->state + ST_TIES;
  a.tie_gap = NEAR_TIE_GAP;
  a.depth_limit = adaptive(c) ? m->state + ST_DLIM : nullptr;
  return SUB_OK;
}

// One decode cycle on the compute stream (capturable): draft D levels,
// verify the tree, accept, compact, advance.
static int32_t enqueue_cycle(sub_model* m, const sub_decode_cfg& c) {
  const sub_model_desc& d = m->d;
  const int k = c.width, D = c.depth;
  const int n_tree = 1 + D * k;
  const int A = d.max_depth + 1;
  sub_tree tr = m->tree;
  tr.width = k;
  tr.max_depth = d.max_depth;
  SUB_CUDA_TRY(mark(m->ev_cyc[0], m->s_main));
  SUB_TRY(begin_target_pass(m));
  // ---- draft ----
  // With verify reuse the draft forward of a level is split at layer R =
  // n_resident: the new nodes' leading part (layers < R, the resident layers
  // the target shares) runs right after the expansion that made them and
  // leaves their residual stream in xsave, and the level's own pass starts
  // from there.  The verify then starts at layer R too.
  const bool reuse = reuses(m, c);
  const int R = d.n_resident;
  auto rows_of = [&](int lvl) {
    const int s0 = lvl == 0 ? 0 : 1 + (lvl - 1) * k;
    const int M = lvl == 0 ? 1 : k;
    FwdRows r{};
    r.tokens = tr.token + s0;
    r.n = M;
    r.slot0 = s0;
    r.depth = tr.depth + s0;
    r.anc = tr.anc + (size_t)s0 * A;
    r.anc_stride = A;
    r.n_slots = s0 + M;
    r.base_dev = m->state + ST_N;
    r.keys_hint = d.max_seq;
    return r;
  };
  auto lead = [&](int lvl) -> int32_t {   // layers [0, R) of level lvl's rows into xsave
    FwdRows r = rows_of(lvl);
    r.layer_end = R;
    r.x_out = m->xsave;
    return forward(m, true, r, nullptr, false);
  };
  if (reuse) SUB_TRY(lead(0));
  // one level: the draft forward over its rows, the expansion into the next
  // level and, with adaptive depth, the decision to go on (next: the next
  // level's conditional node when the cycle is captured)
  auto level = [&](int lvl, cudaGraphConditionalHandle next, int has_next) -> int32_t {
    const int M = lvl == 0 ? 1 : k;
    FwdRows r = rows_of(lvl);
    if (reuse) {
      r.layer0 = R;
      r.x_in = m->xsave;
    }
    SUB_TRY(forward(m, true, r, m->logits, false));
    ExpandArgs e{};
    e.logits = m->logits;
    e.V = d.vocab;
    e.temp = c.draft_temp;
    e.tree = tr;
    e.level = lvl;
    e.k_prev = M;
    e.n_chunks = expand_pick_chunks(M, d.vocab);
    const size_t parts = (size_t)M * e.n_chunks;
    if (parts * MAX_WIDTH > m->part_keys || parts * 2 > m->part_floats)
      return fail(SUB_EINVAL, "expand scratch too small");
    e.part_key = m->part_key;
    e.part_max = m->part_f;
    e.part_sum = m->part_f + parts;
    e.counter = m->counters;
    SUB_TRY(launch_expand(e, m->s_main));
    if (reuse) SUB_TRY(lead(lvl + 1));
    if (adaptive(c))
      SUB_CUDA_TRY(launch_k(adapt_kernel, dim3(1), dim3(32), 0, m->s_main, (const float*)tr.score,
                            1 + lvl * k, k, c.stop_logp, m->state, lvl, next, has_next));
    return SUB_OK;
  };
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  SUB_CUDA_TRY(cudaStreamIsCapturing(m->s_main, &cs));
  const bool captured = cs == cudaStreamCaptureStatusActive;
  if (!adaptive(c)) {
    for (int lvl = 0; lvl < D; ++lvl) SUB_TRY(level(lvl, 0, 0));
  } else if (!captured) {
    // eager: ask the device after every level whether to go on
    for (int lvl = 0; lvl < D; ++lvl) {
      SUB_TRY(level(lvl, 0, 0));
      if (lvl + 1 == D) break;
      SUB_CUDA_TRY(cudaMemcpyAsync(m->host_state, m->state, ST_COUNT * 4, cudaMemcpyDeviceToHost,
                                   m->s_main));
      SUB_CUDA_TRY(cudaStreamSynchronize(m->s_main));
      if (!m->host_state[ST_CONT]) break;
    }
  } else {
    // captured: levels 1 .. D-1 are conditional (IF) nodes of the cycle's graph;
    // each level's adapt kernel opens or closes the next one (handles default to
    // closed at every launch), and a level's body is captured on a side stream
    cudaGraph_t g = nullptr;
    SUB_CUDA_TRY(cudaStreamGetCaptureInfo(m->s_main, &cs, nullptr, &g, nullptr, nullptr, nullptr));
    std::vector<cudaGraphConditionalHandle> h(D, 0);
    for (int lvl = 1; lvl < D; ++lvl)
      SUB_CUDA_TRY(cudaGraphConditionalHandleCreate(&h[lvl], g, 0, cudaGraphCondAssignDefault));
    SUB_TRY(level(0, D > 1 ? h[1] : 0, D > 1));
    for (int lvl = 1; lvl < D; ++lvl) {
      const cudaGraphNode_t* deps = nullptr;
      size_t nd = 0;
      SUB_CUDA_TRY(cudaStreamGetCaptureInfo(m->s_main, &cs, nullptr, &g, &deps, nullptr, &nd));
      cudaGraphNodeParams p{};
      p.type = cudaGraphNodeTypeConditional;
      p.conditional.handle = h[lvl];
      p.conditional.type = cudaGraphCondTypeIf;
      p.conditional.size = 1;
      cudaGraphNode_t node = nullptr;
      SUB_CUDA_TRY(cudaGraphAddNode(&node, g, deps, nullptr, nd, &p));
      SUB_CUDA_TRY(cudaStreamUpdateCaptureDependencies(m->s_main, &node, nullptr, 1,
                                                       cudaStreamSetCaptureDependencies));
      cudaGraph_t body = p.conditional.phGraph_out[0];
      SUB_CUDA_TRY(cudaStreamBeginCaptureToGraph(m->s_cond, body, nullptr, nullptr, 0,
                                                 cudaStreamCaptureModeRelaxed));
      std::swap(m->s_main, m->s_cond);
      const int32_t st_level = level(lvl, lvl + 1 < D ? h[lvl + 1] : 0, lvl + 1 < D);
      std::swap(m->s_main, m->s_cond);
      cudaGraph_t out = nullptr;
      const cudaError_t ee = cudaStreamEndCapture(m->s_cond, &out);
      SUB_TRY(st_level);
      if (ee != cudaSuccess)
        return fail(SUB_ECUDA, std::string("capture of a conditional draft level: ") +
                                   cudaGetErrorString(ee));
      m->cond_kernels += count_kernels(out);
    }
  }
  // ---- verify ----
  SUB_CUDA_TRY(mark(m->ev_cyc[1], m->s_main));
  FwdRows v{};
  v.tokens = tr.token;
  v.n = n_tree;
  v.slot0 = 0;
  v.depth = tr.depth;
  v.anc = tr.anc;
  v.anc_stride = A;
  v.n_slots = n_tree;
  v.base_dev = m->state + ST_N;
  v.keys_hint = d.max_seq;
  if (reuse) {   // layers < R of every tree node were computed by the draft
    v.layer0 = R;
    v.x_in = m->xsave;
  }
  SUB_TRY(forward(m, false, v, m->logits, false));
  SUB_TRY(end_target_pass(m));
  SUB_CUDA_TRY(mark(m->ev_cyc[2], m->s_main));
  // ---- accept, compact, advance ----
  AcceptArgs a;
  SUB_TRY(accept_args(m, c, n_tree, a));
  SUB_TRY(launch_accept(a, m->s_main));
  CompactArgs cp{};
  cp.k = m->kpool;
  cp.v = m->vpool;
  cp.page_table = m->page_table;
  cp.n_layers = d.n_layers;
  cp.n_heads_kv = d.n_heads_kv;
  cp.head_dim = d.head_dim;
  cp.page_size = m->page_size;
  cp.n_pages = m->n_pages;
  cp.root_pos_dev = m->state + ST_N;
  cp.accepted = m->accepted;
  cp.n_accepted = m->state + ST_NACC;
  cp.max_accept = D;
  SUB_TRY(launch_compact(cp, m->s_main));
  SUB_CUDA_TRY(launch_k(advance_kernel, dim3(1), dim3(1), 0, m->s_main, m->state, tr.token));
  return SUB_OK;
}

static bool same_cfg(const sub_decode_cfg& a, const sub_decode_cfg& b) {
  return a.depth == b.depth && a.width == b.width && a.draft_temp == b.draft_temp &&
         a.mode == b.mode && a.target_temp == b.target_temp && a.seed == b.seed &&
         std::memcmp(&a.stop_logp, &b.stop_logp, sizeof(float)) == 0 &&
         (a.verify_reuse != 0) == (b.verify_reuse != 0);
}

static int32_t check_cfg(const sub_model* m, const sub_decode_cfg& c) {
  const sub_model_desc& d = m->d;
  SUB_CHECK_ARG(c.depth >= 0 && c.depth <= d.max_depth, "depth beyond the model's max_depth");
  SUB_CHECK_ARG(c.width >= 1 && c.width <= d.max_width, "width beyond the model's max_width");
  SUB_CHECK_ARG(c.depth == 0 || c.draft_temp > 0.f, "draft_temp must be positive");
  SUB_CHECK_ARG(c.mode == 0 || c.mode == 1, "mode must be 0 or 1");
  SUB_CHECK_ARG(c.mode == 0 || c.target_temp > 0.f, "target_temp must be positive");
  return SUB_OK;
}

// Capture one decode cycle for cfg (once per configuration).
static int32_t ensure_graph(sub_model* m, const sub_decode_cfg& c) {
  if (m->graph && same_cfg(m->graph_cfg, c)) return SUB_OK;
  if (m->graph) {
    cudaGraphExecDestroy(m->graph);
    m->graph = nullptr;
  }
  cudaGraph_t g = nullptr;
  m->cond_kernels = 0;
  SUB_CUDA_TRY(cudaStreamBeginCapture(m->s_main, cudaStreamCaptureModeThreadLocal));
  const int32_t s = enqueue_cycle(m, c);
  const cudaError_t e = cudaStreamEndCapture(m->s_main, &g);
  if (s != SUB_OK) {
    if (g) cudaGraphDestroy(g);
    return s;
  }
  if (e != cudaSuccess) return fail(SUB_ECUDA, std::string("end capture: ") + cudaGetErrorString(e));
  // with adaptive depth: the count when every conditional level runs
  const int64_t kernels = count_kernels(g) + m->cond_kernels;
  const cudaError_t ie = cudaGraphInstantiate(&m->graph, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) {
    m->graph = nullptr;
    return fail(SUB_ECUDA, std::string("graph instantiate: ") + cudaGetErrorString(ie));
  }
  m->graph_cfg = c;
  m->graph_kernels = kernels;
  return SUB_OK;
}

// Order the model's compute stream after `user`, and `user` after it.
static int32_t join_in(sub_model* m, cudaStream_t user) {
  SUB_CUDA_TRY(cudaEventRecord(m->ev_t0, user));
  SUB_CUDA_TRY(cudaStreamWaitEvent(m->s_main, m->ev_t0, 0));
  return SUB_OK;
}
static int32_t join_out(sub_model* m, cudaStream_t user) {
  SUB_CUDA_TRY(cudaEventRecord(m->ev_t1, m->s_main));
  SUB_CUDA_TRY(cudaStreamWaitEvent(user, m->ev_t1, 0));
  return SUB_OK;
}

// Bounded pipeline waits that ran out so far on this device (all kernels).
static int32_t timeouts_now(unsigned int* out) {
  unsigned int a = 0, b = 0;
  SUB_TRY(gemv_tma_timeouts(&a));
  SUB_TRY(gemm_tc_timeouts(&b));
  *out = a + b;
  return SUB_OK;
}
static int32_t check_timeouts(const sub_model* m) {
  unsigned int now = 0;
  SUB_TRY(timeouts_now(&now));
  if (now != m->timeouts0)
    return fail(SUB_ETIMEOUT, std::to_string(now - m->timeouts0) +
                                  " bounded pipeline wait(s) ran out since the prefill: the "
                                  "emitted tokens are not to be trusted");
  return SUB_OK;
}

// Device time between two marks (ms), or a negative value when it cannot be
// read (the error is cleared).
static double span_ms(cudaEvent_t a, cudaEvent_t b) {
  float ms = 0.f;
  if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
    cudaGetLastError();
    return -1e30;
  }
  return ms;
}

static int32_t prefill_impl(sub_model* m, const int32_t* prompt_host, int32_t n_prompt,
                            const sub_decode_cfg& c) {
  const sub_model_desc& d = m->d;
  const cudaStream_t st = m->s_main;
  SUB_CHECK_ARG(n_prompt >= 1 && n_prompt <= d.max_prompt && n_prompt < d.max_seq,
                "n_prompt out of range");
  for (int i = 0; i < n_prompt; ++i)
    SUB_CHECK_ARG(prompt_host[i] >= 0 && prompt_host[i] < d.vocab, "prompt token out of range");
  SUB_TRY(check_cfg(m, c));
  // the prompt goes through pinned staging so the copy is a true async H2D
  SUB_CUDA_TRY(cudaStreamSynchronize(st));
  SUB_TRY(timeouts_now(&m->timeouts0));
  std::memcpy(m->host_prompt, prompt_host, (size_t)n_prompt * 4);
  SUB_CUDA_TRY(cudaMemcpyAsync(m->rows_tok, m->host_prompt, (size_t)n_prompt * 4,
                               cudaMemcpyHostToDevice, st));
  int32_t init[ST_COUNT] = {0};
  init[ST_N] = n_prompt - 1;   // the prefill's last row predicts position n_prompt
  std::memcpy(m->host_state, init, sizeof(init));
  SUB_CUDA_TRY(cudaMemcpyAsync(m->state, m->host_state, sizeof(init), cudaMemcpyHostToDevice, st));
  FwdRows p{};
  p.tokens = m->rows_tok;
  p.n = n_prompt;
  p.slot0 = 0;
  p.n_slots = n_prompt;
  p.base = 0;
  p.keys_hint = n_prompt;
  SUB_TRY(begin_target_pass(m));
  SUB_TRY(forward(m, false, p, m->logits, true));
  SUB_TRY(end_target_pass(m));
  AcceptArgs a;
  SUB_TRY(accept_args(m, c, 1, a));
  a.hist = nullptr;
  SUB_TRY(launch_accept(a, st));
  SUB_CUDA_TRY(launch_k(advance_kernel, dim3(1), dim3(1), 0, st, m->state, m->tree.token));
  SUB_CUDA_TRY(cudaMemsetAsync(m->hist, 0, (d.max_depth + 1) * 4, st));
  m->n_prompt = n_prompt;
  m->cycles = 0;
  m->max_emit = d.max_seq - n_prompt;
  return SUB_OK;
}

static int32_t decode_impl(sub_model* m, const sub_decode_cfg& c, int32_t n_cycles) {
  SUB_TRY(check_cfg(m, c));
  SUB_CHECK_ARG(n_cycles >= 0, "n_cycles must be >= 0");
  SUB_CHECK_ARG(m->n_prompt > 0, "sub_prefill must run first");
  SUB_CHECK_ARG((int64_t)(m->cycles + n_cycles) * (c.depth + 1) + 1 <= m->max_emit ||
                    n_cycles <= 1,
                "n_cycles could overflow max_seq");
  if (c.use_graph) SUB_TRY(ensure_graph(m, c));
  for (int i = 0; i < n_cycles; ++i) {
    if (c.use_graph) SUB_CUDA_TRY(cudaGraphLaunch(m->graph, m->s_main));
    else SUB_TRY(enqueue_cycle(m, c));
  }
  m->cycles += n_cycles;
  return SUB_OK;
}

static int32_t read_state(sub_model* m) {
  SUB_CUDA_TRY(cudaMemcpyAsync(m->host_state, m->state, ST_COUNT * 4, cudaMemcpyDeviceToHost,
                               m->s_main));
  SUB_CUDA_TRY(cudaStreamSynchronize(m->s_main));
  if (m->host_state[ST_EMITTED] > m->out_cap)
    return fail(SUB_ECUDA, "decode state corrupted (emitted overflow)");
  return SUB_OK;
}

extern "C" int32_t sub_prefill(sub_model* m, const int32_t* prompt_host, int32_t n_prompt,
                               const sub_decode_cfg* cfg, void* stream) {
  SUB_CHECK_ARG(m && prompt_host && cfg, "null pointer");
  SUB_TRY(join_in(m, as_stream(stream)));
  SUB_TRY(prefill_impl(m, prompt_host, n_prompt, *cfg));
  return join_out(m, as_stream(stream));
}

extern "C" int32_t sub_decode_cycles(sub_model* m, const sub_decode_cfg* cfg, int32_t n_cycles,
                                     void* stream) {
  SUB_CHECK_ARG(m && cfg, "null pointer");
  SUB_TRY(join_in(m, as_stream(stream)));
  SUB_TRY(decode_impl(m, *cfg, n_cycles));
  return join_out(m, as_stream(stream));
}

extern "C" int32_t sub_decode_read(sub_model* m, int32_t* out_host, int32_t n, int32_t* emitted,
                                   int64_t* cycles) {
  SUB_CHECK_ARG(m, "null pointer");
  SUB_TRY(read_state(m));
  const int32_t tstat = check_timeouts(m);
  const int e = m->host_state[ST_EMITTED];
  if (emitted) *emitted = e;
  if (cycles) *cycles = m->cycles;
  if (out_host && n > 0) {
    const int cnt = std::min(n, e);
    SUB_CUDA_TRY(cudaMemcpy(out_host, m->out_tokens, (size_t)cnt * 4, cudaMemcpyDeviceToHost));
  }
  return tstat;
}

extern "C" int32_t sub_cycle_info(sub_model* m, const sub_decode_cfg* cfg,
                                  int64_t* kernels_per_cycle, int64_t* h2d_bytes_per_cycle) {
  SUB_CHECK_ARG(m && cfg, "null pointer");
  SUB_TRY(check_cfg(m, *cfg));
  sub_decode_cfg c = *cfg;
  c.use_graph = 1;
  SUB_TRY(ensure_graph(m, c));
  if (kernels_per_cycle) *kernels_per_cycle = m->graph_kernels;
  if (h2d_bytes_per_cycle) {
    int64_t b = 0;
    for (int i = 0; i < 7; ++i) b += (int64_t)m->mat_bytes[i];
    *h2d_bytes_per_cycle = b * m->n_off;
  }
  return SUB_OK;
}

extern "C" int32_t sub_generate(sub_model* m, const int32_t* prompt_host, int32_t n_prompt,
                                int32_t n_new, const sub_decode_cfg* cfg, int32_t* out_tokens_host,
                                sub_stats* stats) {
  SUB_CHECK_ARG(m && prompt_host && cfg && out_tokens_host, "null pointer");
  const sub_model_desc& d = m->d;
  const sub_decode_cfg c = *cfg;
  SUB_CHECK_ARG(n_new >= 1 && (int64_t)n_prompt + n_new <= d.max_seq, "n_prompt + n_new > max_seq");
  const cudaStream_t st = m->s_main;
  SUB_CUDA_TRY(cudaStreamSynchronize(st));
  // a new configuration's cycle graph is captured before the timed spans, so
  // t_prefill_ms and t_decode_ms are device time only
  SUB_TRY(check_cfg(m, c));
  if (c.use_graph) SUB_TRY(ensure_graph(m, c));
  SUB_CUDA_TRY(cudaEventRecord(m->ev_g0, st));
  SUB_TRY(prefill_impl(m, prompt_host, n_prompt, c));
  SUB_CUDA_TRY(cudaEventRecord(m->ev_g1, st));
  SUB_TRY(read_state(m));
  int emitted = m->host_state[ST_EMITTED];
  double t_draft = 0.0, t_verify = 0.0, t_unhidden = 0.0, t_copy = 0.0;
  while (emitted < n_new) {
    SUB_TRY(decode_impl(m, c, 1));
    SUB_TRY(read_state(m));
    emitted = m->host_state[ST_EMITTED];
    // this cycle's phase times (the marks of the cycle just synchronised)
    t_draft += span_ms(m->ev_cyc[0], m->ev_cyc[1]);
    t_verify += span_ms(m->ev_cyc[1], m->ev_cyc[2]);
    if (m->n_off > 0) {
      const double c = span_ms(m->ev_cyc[0], m->ev_tstaged[m->n_off - 1]);
      t_copy = (c < -1e29 || t_copy < 0.0) ? -1.0 : t_copy + c;
    }
    for (int j = 0; j < m->n_off; ++j) {
      const double w = span_ms(m->ev_ready[j], m->ev_tstaged[j]);   // < 0: copy was early
      t_unhidden = (w < -1e29 || t_unhidden < 0.0) ? -1.0 : t_unhidden + std::max(0.0, w);
    }
  }
  SUB_CUDA_TRY(cudaEventRecord(m->ev_g2, st));
  SUB_CUDA_TRY(cudaMemcpyAsync(m->host_out, m->out_tokens, (size_t)n_new * 4,
                               cudaMemcpyDeviceToHost, st));
  SUB_CUDA_TRY(cudaStreamSynchronize(st));
  std::memcpy(out_tokens_host, m->host_out, (size_t)n_new * 4);
  if (stats) {
    float t_prefill = 0.f, t_decode = 0.f;
    SUB_CUDA_TRY(cudaEventElapsedTime(&t_prefill, m->ev_g0, m->ev_g1));
    SUB_CUDA_TRY(cudaEventElapsedTime(&t_decode, m->ev_g1, m->ev_g2));
    std::memset(stats, 0, sizeof(*stats));
    stats->cycles = m->cycles;
    stats->emitted = n_new;
    stats->tau = m->cycles ? (double)(emitted - 1) / (double)m->cycles : 0.0;
    stats->t_prefill_ms = t_prefill;
    stats->t_decode_ms = t_decode;
    std::vector<int32_t> h(d.max_depth + 1);
    SUB_CUDA_TRY(cudaMemcpy(h.data(), m->hist, h.size() * 4, cudaMemcpyDeviceToHost));
    for (int i = 0; i <= std::min(d.max_depth, 64); ++i) stats->accept_hist[i] = h[i];
    stats->t_draft_ms = t_draft >= 0.0 ? t_draft : -1.0;
    stats->t_verify_ms = t_verify >= 0.0 ? t_verify : -1.0;
    stats->t_copy_unhidden_ms = t_unhidden >= 0.0 ? t_unhidden : -1.0;
    stats->t_copy_ms = t_copy >= 0.0 ? t_copy : -1.0;
    stats->near_tie_events = m->host_state[ST_TIES];
    stats->drafted_levels = adaptive(c) ? m->host_state[ST_LEVELS] : m->cycles * c.depth;
  }
  return check_timeouts(m);
}
