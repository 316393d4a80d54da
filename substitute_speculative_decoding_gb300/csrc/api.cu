// C ABI entry points for the kernels (the model and generate calls live in
// model.cu): argument checks, temporary scratch, launch.
#include <algorithm>
#include <cstdlib>
#include <mutex>
#include "attn.cuh"
#include "gemm.cuh"
#include "tree.cuh"

namespace sub {

static thread_local std::string g_last_error;

bool env_flag(const char* name, bool dflt) {
  const char* e = getenv(name);
  if (!e || !e[0]) return dflt;
  return e[0] != '0';
}
bool pdl_enabled() {
  static const bool on = env_flag("SUB_PDL", true);
  return on;
}

bool fault_injected(const char* kind, int index) {
  const char* e = getenv("SUB_FAULT");
  if (!e || !e[0]) return false;
  const size_t n = strlen(kind);
  if (strncmp(e, kind, n) != 0) return false;
  if (e[n] == '\0') return true;                    // every event of this kind
  if (e[n] != ':') return false;
  return atoi(e + n + 1) == index;                  // only the given one
}

void set_error(const std::string& msg) { g_last_error = msg; }
int32_t fail(int32_t code, const std::string& msg) {
  g_last_error = msg;
  return code;
}
int32_t check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SUB_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return SUB_OK;
}

// Temporary device memory on a stream (freed in stream order).
struct StreamScratch {
  void* p = nullptr;
  cudaStream_t st;
  explicit StreamScratch(cudaStream_t s) : st(s) {}
  int32_t alloc(size_t bytes) {
    if (bytes == 0) return SUB_OK;
    const cudaError_t e = cudaMallocAsync(&p, bytes, st);
    if (e != cudaSuccess) {
      p = nullptr;
      return fail(SUB_ENOMEM, std::string("cudaMallocAsync: ") + cudaGetErrorString(e));
    }
    return SUB_OK;
  }
  ~StreamScratch() {
    if (p) cudaFreeAsync(p, st);
  }
};

}  // namespace sub

using namespace sub;

extern "C" const char* sub_last_error(void) { return g_last_error.c_str(); }
extern "C" const char* sub_version(void) { return "0.1 sm_103a"; }

extern "C" int32_t sub_pipeline_timeouts(uint32_t* out) {
  SUB_CHECK_ARG(out, "null pointer");
  unsigned int a = 0, b = 0;
  SUB_TRY(gemv_tma_timeouts(&a));
  SUB_TRY(gemm_tc_timeouts(&b));
  *out = a + b;
  return SUB_OK;
}

extern "C" int32_t sub_bounded_wait_check(uint32_t max_polls) {
  SUB_CHECK_ARG(max_polls >= 1 && max_polls <= (1u << 20), "max_polls must be in [1, 2^20]");
  uint32_t polls = 1;
  SUB_TRY(bounded_wait_selftest(max_polls, &polls));
  if (polls == 0)
    return fail(SUB_ETIMEOUT, "bounded wait gave up after " + std::to_string(max_polls) +
                                  " polls; the kernel ended normally");
  return SUB_OK;
}

static int32_t matmul_public(const sub_bf16* X, int64_t M, bool w4, const void* W,
                             const sub_bf16* scale, const sub_bf16* zero, int64_t N, int64_t K,
                             sub_bf16* Y, void* stream, int bits = 4) {
  SUB_CHECK_ARG(X && W && Y, "null pointer");
  SUB_CHECK_ARG(M >= 1 && N >= 1 && K >= 8 && K % 8 == 0, "bad sizes (K % 8 == 0 required)");
  SUB_CHECK_ARG(M < (1 << 24) && N < (1 << 30) && K < (1 << 30), "sizes too large");
  SUB_CHECK_ARG(aligned16(X) && aligned16(W), "X and W must be 16-byte aligned");
  GemvArgs a{};
  a.X = X;
  a.M = (int)M;
  a.K = (int)K;
  a.ldx = (int)K;
  a.W[0] = W;
  a.S[0] = scale;
  a.Z[0] = zero;
  a.seg_end[0] = (int)N;
  a.n_seg = 1;
  a.N = (int)N;
  a.Y = Y;
  a.ldy = (int)N;
  a.bits = w4 ? bits : 0;
  const cudaStream_t st = as_stream(stream);
  StreamScratch scratch(st);
  // split scratch: partial sums of K splits (register-streamed kernel) or of
  // blocks shared by several CTAs (TMA kernel), and one counter per row unit
  const int ks = M <= 16 ? gemv_ksplit(a, w4, EPI_BF16) : 1;
  size_t tma_floats = M <= 16 ? gemv_tma_scratch_floats(a, w4, EPI_BF16)
                              : gemm_tc_scratch_floats(a, w4, EPI_BF16);
  if (M > 16 && M <= 32 && w4)   // the four-tile TMA GEMV may take it (int4)
    tma_floats = std::max(tma_floats, gemv_tma_scratch_floats(a, w4, EPI_BF16));
  if (ks > 1 || tma_floats > 0) {
    // row units of 16, or weight tiles x token tiles of the tensor-core GEMM
    const int units = (int)std::max<int64_t>((N + 15) / 16, ((N + 127) / 128) * ((M + 255) / 256));
    a.split_cap = std::max((size_t)units * ks * 4 * 128, tma_floats);
    a.split_cnt_cap = units;
    SUB_TRY(scratch.alloc(a.split_cap * 4 + (size_t)units * 4));
    a.split_part = reinterpret_cast<float*>(scratch.p);
    a.split_cnt = reinterpret_cast<unsigned int*>(a.split_part + a.split_cap);
    SUB_CUDA_TRY(cudaMemsetAsync(a.split_cnt, 0, (size_t)units * 4, st));
  }
  return launch_matmul(a, w4, EPI_BF16, st);
}

extern "C" int32_t sub_w4_gemm(const sub_bf16* X, int64_t M, const uint8_t* q,
                               const sub_bf16* scale, const sub_bf16* zero, int64_t N, int64_t K,
                               int32_t group, sub_bf16* Y, void* stream) {
  if (group != 64) return fail(SUB_EUNSUPPORTED, "group must be 64");
  SUB_CHECK_ARG(scale && zero, "null pointer");
  return matmul_public(X, M, true, q, scale, zero, N, K, Y, stream);
}

extern "C" int32_t sub_wq_gemm(const sub_bf16* X, int64_t M, const uint8_t* q,
                               const sub_bf16* scale, const sub_bf16* zero, int64_t N, int64_t K,
                               int32_t group, int32_t bits, sub_bf16* Y, void* stream) {
  if (group != 64) return fail(SUB_EUNSUPPORTED, "group must be 64");
  SUB_CHECK_ARG(bits == 2 || bits == 3 || bits == 4, "bits must be 2, 3 or 4");
  SUB_CHECK_ARG(X && q && scale && zero && Y, "null pointer");
  if (M <= 16 || bits == 4) return matmul_public(X, M, true, q, scale, zero, N, K, Y, stream, bits);
  // wider products of 2- and 3-bit codes: dequantise into scratch, then the
  // bf16 tensor-core GEMM (the same bf16((q - z) * s) values the oracle uses)
  SUB_CHECK_ARG(N >= 1 && K >= 8 && K % 8 == 0 && N < (1 << 30) && K < (1 << 30), "bad sizes");
  const cudaStream_t st = as_stream(stream);
  StreamScratch deq(st);
  SUB_TRY(deq.alloc((size_t)N * (size_t)K * 2));
  sub_bf16* Wd = reinterpret_cast<sub_bf16*>(deq.p);
  SUB_TRY(sub_wq_dequant(q, scale, zero, N, K, group, bits, Wd, stream));
  return matmul_public(X, M, false, Wd, nullptr, nullptr, N, K, Y, stream);
}

extern "C" int32_t sub_bf16_gemm(const sub_bf16* X, int64_t M, const sub_bf16* W, int64_t N,
                                 int64_t K, sub_bf16* Y, void* stream) {
  return matmul_public(X, M, false, W, nullptr, nullptr, N, K, Y, stream);
}

extern "C" int32_t sub_tree_attn(const sub_bf16* Q, int32_t n_q, int32_t n_heads_q,
                                 const sub_kv_cache* kv, int32_t layer, int64_t n_prefix,
                                 int64_t tree_base, int32_t n_slots, const int32_t* anc,
                                 int32_t anc_stride, const int32_t* depth, float softmax_scale,
                                 sub_bf16* O, void* stream) {
  SUB_CHECK_ARG(kv && Q && O, "null pointer");
  SUB_CHECK_ARG(n_q >= 0, "n_q must be >= 0");
  SUB_CHECK_ARG(layer >= 0 && layer < kv->n_layers, "layer out of range");
  SUB_CHECK_ARG(n_prefix >= 0 && tree_base >= 0, "negative position");
  SUB_CHECK_ARG(n_prefix <= kv->capacity && tree_base + n_slots <= kv->capacity,
                "keys beyond the cache capacity");
  SUB_CHECK_ARG(!anc || (depth && anc_stride >= 1), "anc needs depth and anc_stride");
  SUB_CHECK_ARG(anc || n_slots >= n_q, "chain mode needs n_slots >= n_q");
  SUB_CHECK_ARG(aligned16(Q) && aligned16(O) && aligned16(kv->k) && aligned16(kv->v),
                "tensors must be 16-byte aligned");
  AttnArgs a{};
  a.Q = Q;
  a.O = O;
  a.n_q = n_q;
  a.n_heads_q = n_heads_q;
  a.n_heads_kv = kv->n_heads_kv;
  a.head_dim = kv->head_dim;
  a.k = kv->k;
  a.v = kv->v;
  a.page_table = kv->page_table;
  a.page_size = kv->page_size;
  a.n_pages = kv->n_pages;
  a.layer = layer;
  a.n_prefix = n_prefix;
  a.tree_base = tree_base;
  a.n_slots = n_slots;
  a.anc = anc;
  a.anc_stride = anc_stride;
  a.depth = depth;
  a.chain_slot0 = 0;
  a.scale = softmax_scale;
  if (n_q == 0) return SUB_OK;
  SUB_CHECK_ARG(n_heads_q >= 1 && kv->n_heads_kv >= 1 && n_heads_q % kv->n_heads_kv == 0,
                "Hq must be a multiple of Hkv");
  const cudaStream_t st = as_stream(stream);
  const int splits = attn_pick_splits(a, (int)(n_prefix + n_slots), true);
  StreamScratch scratch(st);
  const size_t xf = attn_xpart_floats(a, splits), xc = attn_xcnt_count(a, splits);
  if (xf) {   // two clusters per row block: their partials and counters
    SUB_TRY(scratch.alloc(xf * 4 + xc * 4));
    const size_t rows = xf / (a.head_dim + 2);
    a.xpart = reinterpret_cast<float*>(scratch.p);
    a.xm = a.xpart + rows * a.head_dim;
    a.xl = a.xm + rows;
    a.xcnt = reinterpret_cast<unsigned int*>(a.xl + rows);
    SUB_CUDA_TRY(cudaMemsetAsync(a.xcnt, 0, xc * 4, st));
  }
  return launch_tree_attn(a, splits, st);
}

extern "C" int32_t sub_draft_expand(const float* logits, int64_t V, float temperature,
                                    const sub_tree* tree, int32_t level, void* stream) {
  SUB_CHECK_ARG(logits && tree && tree->token && tree->parent && tree->depth && tree->score &&
                    tree->anc,
                "null pointer");
  SUB_CHECK_ARG(tree->max_depth >= 1, "tree depth must be >= 1");
  ExpandArgs a{};
  a.logits = logits;
  a.V = V;
  a.temp = temperature;
  a.tree = *tree;
  a.level = level;
  a.k_prev = level == 0 ? 1 : tree->width;
  a.n_chunks = expand_pick_chunks(a.k_prev, V);
  const cudaStream_t st = as_stream(stream);
  StreamScratch scratch(st);
  const size_t parts = (size_t)a.k_prev * a.n_chunks;
  SUB_TRY(scratch.alloc(expand_scratch_bytes(a.k_prev, a.n_chunks, tree->width)));
  a.part_key = reinterpret_cast<unsigned long long*>(scratch.p);
  a.part_max = reinterpret_cast<float*>(a.part_key + parts * MAX_WIDTH);
  a.part_sum = a.part_max + parts;
  a.counter = reinterpret_cast<unsigned int*>(a.part_sum + parts);
  SUB_CUDA_TRY(cudaMemsetAsync(a.counter, 0, sizeof(unsigned int), st));
  return launch_expand(a, st);
}

static int32_t accept_args(const float* logits, const sub_tree* tree, int32_t n_nodes, int64_t V,
                           int32_t mode, float temperature, uint64_t seed, int64_t root_pos,
                           int32_t* accepted_slots, int32_t* n_accepted, int32_t* bonus_token,
                           AcceptArgs* a) {
  SUB_CHECK_ARG(logits && tree && accepted_slots && n_accepted && bonus_token, "null pointer");
  SUB_CHECK_ARG(n_nodes >= 1 && n_nodes <= 1 + tree->max_depth * tree->width,
                "n_nodes out of range");
  SUB_CHECK_ARG(root_pos >= 0, "root_pos must be >= 0");
  *a = AcceptArgs{};
  a->logits = logits;
  a->V = V;
  a->tree = *tree;
  a->n_nodes = n_nodes;
  a->mode = mode;
  a->temp = temperature;
  a->seed = seed;
  a->root_pos = root_pos;
  a->n_chunks = accept_pick_chunks(n_nodes, V);
  a->accepted = accepted_slots;
  a->n_accepted = n_accepted;
  a->bonus = bonus_token;
  return SUB_OK;
}

// Scratch layout of one accept call: part keys, then the counter (64 bytes),
// then the choice array when the caller gives none.
static size_t accept_scratch_bytes(const AcceptArgs& a, bool own_choice) {
  return (size_t)a.n_nodes * a.n_chunks * 8 + 64 + (own_choice ? (size_t)a.n_nodes * 4 : 0);
}
static int32_t accept_on(AcceptArgs& a, void* scratch, int32_t* choice, cudaStream_t st) {
  const size_t key_bytes = (size_t)a.n_nodes * a.n_chunks * 8;
  a.part_key = reinterpret_cast<unsigned long long*>(scratch);
  a.counter = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(scratch) + key_bytes);
  a.choice = choice ? choice
                    : reinterpret_cast<int32_t*>(reinterpret_cast<char*>(scratch) + key_bytes + 64);
  SUB_CUDA_TRY(cudaMemsetAsync(a.counter, 0, sizeof(unsigned int), st));
  return launch_accept(a, st);
}

extern "C" int32_t sub_verify_accept(const float* logits, const sub_tree* tree, int32_t n_nodes,
                                     int64_t V, int32_t mode, float temperature, uint64_t seed,
                                     int64_t root_pos, int32_t* accepted_slots,
                                     int32_t* n_accepted, int32_t* bonus_token, int32_t* choice,
                                     void* stream) {
  AcceptArgs a;
  SUB_TRY(accept_args(logits, tree, n_nodes, V, mode, temperature, seed, root_pos, accepted_slots,
                      n_accepted, bonus_token, &a));
  const cudaStream_t st = as_stream(stream);
  StreamScratch scratch(st);
  SUB_TRY(scratch.alloc(accept_scratch_bytes(a, !choice)));
  return accept_on(a, scratch.p, choice, st);
}

// The fixed scratch of sub_verify_accept_static: one array per device (each
// device's copy of the module has its own), looked up once per device.
static __device__ __align__(256) unsigned char g_accept_scratch[SUB_ACCEPT_STATIC_BYTES];

static int32_t accept_static_base(void** out) {
  constexpr int MAX_DEV = 64;
  static std::mutex mu;
  static void* base[MAX_DEV] = {};
  int dev = 0;
  SUB_CUDA_TRY(cudaGetDevice(&dev));
  SUB_CHECK_ARG(dev >= 0 && dev < MAX_DEV, "device ordinal beyond the static scratch table");
  std::lock_guard<std::mutex> lock(mu);
  if (!base[dev]) SUB_CUDA_TRY(cudaGetSymbolAddress(&base[dev], g_accept_scratch));
  *out = base[dev];
  return SUB_OK;
}

extern "C" int32_t sub_verify_accept_static(const float* logits, const sub_tree* tree,
                                            int32_t n_nodes, int64_t V, int32_t mode,
                                            float temperature, uint64_t seed, int64_t root_pos,
                                            int32_t* accepted_slots, int32_t* n_accepted,
                                            int32_t* bonus_token, int32_t* choice, void* stream) {
  AcceptArgs a;
  SUB_TRY(accept_args(logits, tree, n_nodes, V, mode, temperature, seed, root_pos, accepted_slots,
                      n_accepted, bonus_token, &a));
  SUB_CHECK_ARG(accept_scratch_bytes(a, !choice) <= (size_t)SUB_ACCEPT_STATIC_BYTES,
                "n_nodes too large for the static accept scratch");
  void* base = nullptr;
  SUB_TRY(accept_static_base(&base));
  return accept_on(a, base, choice, as_stream(stream));
}

extern "C" int32_t sub_kv_compact(const sub_kv_cache* kv, int64_t root_pos,
                                  const int32_t* accepted_slots, const int32_t* n_accepted,
                                  int32_t max_accept, void* stream) {
  SUB_CHECK_ARG(kv && accepted_slots && n_accepted, "null pointer");
  SUB_CHECK_ARG(root_pos >= 0 && root_pos + max_accept < kv->capacity, "positions beyond capacity");
  CompactArgs a{};
  a.k = kv->k;
  a.v = kv->v;
  a.page_table = kv->page_table;
  a.n_layers = kv->n_layers;
  a.n_heads_kv = kv->n_heads_kv;
  a.head_dim = kv->head_dim;
  a.page_size = kv->page_size;
  a.n_pages = kv->n_pages;
  a.root_pos = root_pos;
  a.accepted = accepted_slots;
  a.n_accepted = n_accepted;
  a.max_accept = max_accept;
  return launch_compact(a, as_stream(stream));
}
