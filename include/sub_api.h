/*
 * sub_api.h -- C ABI of the SubSpec draft-and-verify decode library (sm_103a).
 *
 * SubSpec (substitute speculative decoding) accelerates a dense decoder that
 * does not fit in GPU memory: the offloaded target layers get 4-bit
 * substitutes kept on the GPU; the draft = the target's own resident layers +
 * the substitutes, sharing the target's KV cache, and it drafts a deep static
 * token tree from temperature-sharpened probabilities; the target verifies the
 * whole tree in one pass and the longest matching path is accepted, so the
 * output equals plain target decoding token for token.
 *   "Speculate Deep and Accurate: Lossless and Training-Free Acceleration for
 *    Offloaded LLMs via Substitute Speculative Decoding" -- abstract and the
 *    summary card (Problem, Approach);
 *   "SubSpec: Using the Target Model's Own Low-Bit Shadow as Its Draft Model"
 *    -- reading report, 2.2 Step 4, 4.1, 6.2 (Leviathan et al.), 6.3 (SpecInfer).
 *
 * Conventions (every entry point):
 *   - returns int32_t status: SUB_OK or a SUB_E* code; nothing aborts or
 *     throws across the ABI; sub_last_error() gives a message for the calling
 *     thread's last failure.
 *   - pointers are DEVICE pointers unless the name ends in _host.  The caller
 *     owns every buffer it passes; the library keeps no caller pointer past the
 *     call except those stored in a sub_model (weights, see sub_model_desc).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Kernel entry points only enqueue work; sub_generate synchronises.
 *   - bf16 tensors are raw uint16 bit patterns (sub_bf16), row-major.
 *   - group must be 64 (SUB_EUNSUPPORTED otherwise).
 */
#ifndef SUB_API_H
#define SUB_API_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t sub_bf16;

enum {
  SUB_OK = 0,
  SUB_EINVAL = 1,        /* bad argument: size, null pointer, alignment */
  SUB_ENOMEM = 2,        /* device or pinned allocation failed */
  SUB_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  SUB_EUNSUPPORTED = 4,  /* valid but not implemented (e.g. group != 64) */
  SUB_ETIMEOUT = 5       /* a bounded device wait gave up */
};

/* Message of the calling thread's last failed call ("" if none). */
const char* sub_last_error(void);

/* Library version string and the compile target, e.g. "0.1 sm_103a". */
const char* sub_version(void);

/* Host-side fault injection for tests (no device fault is ever made): the
 * environment variable SUB_FAULT, read at each call, makes a library call fail
 * as if a CUDA call had failed:
 *   SUB_FAULT=alloc:N  the N-th device allocation of sub_model_create (0-based)
 *                      fails: the call returns SUB_ENOMEM and frees what it
 *                      had allocated;
 *   SUB_FAULT=h2d      every host-to-device copy of streamed originals fails:
 *                      sub_prefill / sub_generate / target forwards return
 *                      SUB_ECUDA; the model stays valid and can be destroyed.
 * Unset (the default) costs one getenv per allocation or copy. */

/* Pipeline waits that ran out on the current device since the library was
 * loaded.  Every wait inside the TMA-streamed GEMV and the tensor-core GEMM
 * (mbarrier phases, the grid-wide counters) is bounded: one that runs out
 * bumps this count and lets the kernel finish with wrong numbers instead of
 * hanging.  A correct run leaves it at 0; a non-zero value means the results
 * of that run are invalid.  *out receives the count. */
int32_t sub_pipeline_timeouts(uint32_t* out);

/* Check of the bounded-wait mechanism itself: one kernel thread waits on an
 * mbarrier that nothing ever arrives on (and no copy targets), polling at most
 * max_polls times (1 .. 2^20), with the same wait routine the pipelines use.
 * The wait gives up, the kernel ends normally and the context stays usable:
 * the call returns SUB_ETIMEOUT (SUB_OK would mean the barrier completed,
 * which cannot happen).  It leaves sub_pipeline_timeouts unchanged. */
int32_t sub_bounded_wait_check(uint32_t max_polls);

/* ------------------------------------------------------------------------ */
/* Int4 substitutes.  The draft replaces each offloaded target layer by a
 * data-free 4-bit copy ("Low-Bit Shadow" report 2.2 Step 4; card, Approach).
 * This library's quantiser: per row n and group g of 64 consecutive inputs
 * along K,  s = bf16(fp32(hi-lo)/15) (s = 1 if that is 0),
 * z = bf16(fp32(-lo)/s),  q = clamp(rint_even(fp32(w/s) + z), 0, 15),
 * dequantised value bf16((q - z) * s).  Layout: q is uint8 [N, ceil(K/64)*32]
 * (byte j of a group: element 2j in the low nibble, 2j+1 in the high nibble;
 * nibbles past K are 0); scale and zero are bf16 [N, ceil(K/64)].          */

/* Quantise W (bf16 [N, K]) into q, scale, zero.  Bit-exact with the rule
 * above.  K >= 1, N >= 1; W rows must be 16-byte aligned (K % 8 == 0). */
int32_t sub_w4_pack(const sub_bf16* W, int64_t N, int64_t K, int32_t group,
                    uint8_t* q, sub_bf16* scale, sub_bf16* zero, void* stream);

/* Dequantise to bf16 W_out [N, K] (a test and debugging aid). */
int32_t sub_w4_dequant(const uint8_t* q, const sub_bf16* scale, const sub_bf16* zero,
                       int64_t N, int64_t K, int32_t group, sub_bf16* W_out, void* stream);

/* Y[M, N] (bf16) = X[M, K] (bf16) . deq(W)^T, fp32 accumulation.
 * M <= 16, and M <= 32 where K % 512 == 0, runs the warp-level GEMV (one
 * pass over the packed weights; the zero point and scale are folded into the
 * fp32 sums, so deq(W) is not rounded to bf16 there, and a row's result does
 * not depend on M).  Larger M runs the tcgen05 tensor-core GEMM, which
 * dequantises each 64-column group to bf16((q - z) * s), the values
 * sub_w4_dequant returns, before the multiply.  K % 8 == 0. */
int32_t sub_w4_gemm(const sub_bf16* X, int64_t M, const uint8_t* q, const sub_bf16* scale,
                    const sub_bf16* zero, int64_t N, int64_t K, int32_t group,
                    sub_bf16* Y, void* stream);

/* Y[M, N] (bf16) = X[M, K] . W[N, K]^T for bf16 weights (resident layers and
 * streamed originals).  Same kernel family the decode path uses. K % 8 == 0. */
int32_t sub_bf16_gemm(const sub_bf16* X, int64_t M, const sub_bf16* W, int64_t N, int64_t K,
                      sub_bf16* Y, void* stream);

/* ------------------------------------------------------------------------ */
/* 2-, 3- and 4-bit substitutes (lower and per-layer mixed precision for the
 * substitute layers: "Low-Bit Shadow" report 5.1 point 2 and 10.1 (2), which
 * leave 2/3-bit substitutes untested; 10.2 (10), precision per layer by
 * sensitivity).  The same quantiser with L = 2^bits - 1 levels in place of 15:
 * s = bf16(fp32(hi-lo)/L) (1 if that is 0), z = bf16(fp32(-lo)/s),
 * q = clamp(rint_even(fp32(w/s) + z), 0, L), dequantised bf16((q - z) * s).
 * q is uint8 [N, ceil(K/64) * 8 * bits]; per 64-element group:
 *   bits 4: 32 bytes, the int4 layout above (sub_w4_* are these calls at 4);
 *   bits 2: 16 bytes, byte j holds elements 4j..4j+3 at bits 0-1, 2-3, 4-5, 6-7;
 *   bits 3: 24 bytes, bytes 0..15 the 2-bit layout of (q & 3), then bit i of
 *           byte 16 + j is q(8j + i) >> 2.
 * Codes past K are 0; scale and zero are bf16 [N, ceil(K/64)].  Arguments,
 * alignment and errors as for the sub_w4_* calls; bits outside {2, 3, 4}
 * returns SUB_EINVAL. */
int32_t sub_wq_pack(const sub_bf16* W, int64_t N, int64_t K, int32_t group, int32_t bits,
                    uint8_t* q, sub_bf16* scale, sub_bf16* zero, void* stream);
int32_t sub_wq_dequant(const uint8_t* q, const sub_bf16* scale, const sub_bf16* zero, int64_t N,
                       int64_t K, int32_t group, int32_t bits, sub_bf16* W_out, void* stream);
/* sub_wq_pack with the zero point optimised by HQQ (the pages' quantiser:
 * "Low-Bit Shadow" report Critique 3 and 6.2; their steps are not given
 * there, these follow the published half-quadratic method).  The min-max
 * scale is kept; per group, starting from the min-max zero z (unrounded),
 * `iters` steps of
 *   q = clamp(rint(w/s + z), 0, L),  r = w - s (q - z),
 *   e = sign(r) max(|r| - |r|^(-1/2) / beta, 0),  z = mean(q - (w - e)/s),
 *   beta = beta * 1.01   (beta starts at 10)
 * keep the zero with the smallest sum |r| (ties: the earlier); it is rounded
 * to bf16 and the codes are formed with it.  Every step is one IEEE fp32
 * operation and the group sums run in one fixed pairwise order, so the
 * result is reproducible bit for bit.  The output is in the sub_wq layouts
 * and dequantises with the same rule.  iters in [1, 1000]; iters = 1 gives
 * the min-max quantiser. */
int32_t sub_wq_pack_hqq(const sub_bf16* W, int64_t N, int64_t K, int32_t group, int32_t bits,
                        int32_t iters, uint8_t* q, sub_bf16* scale, sub_bf16* zero,
                        void* stream);
/* Y[M, N] (bf16) = X[M, K] . deq(W)^T.  M <= 16: the warp-level GEMV with the
 * zero point and scale folded into fp32 sums (2- and 3-bit codes are spread
 * into the int4 word layout in registers or shared memory).  Larger M at 2 or 3 bits:
 * dequantise into stream-ordered scratch (N * K * 2 bytes, SUB_ENOMEM if it
 * cannot be had) and run the bf16 tensor-core GEMM; at 4 bits as sub_w4_gemm. */
int32_t sub_wq_gemm(const sub_bf16* X, int64_t M, const uint8_t* q, const sub_bf16* scale,
                    const sub_bf16* zero, int64_t N, int64_t K, int32_t group, int32_t bits,
                    sub_bf16* Y, void* stream);

/* ------------------------------------------------------------------------ */
/* Shared paged KV cache.  The draft attends over the target's committed KV
 * ("Low-Bit Shadow" report 4.1 point 2: draft and target see the same
 * attention context; card, measured effects: shared KV-cache).
 * Pools k and v hold, for each layer l and physical page p,
 * [n_heads_kv][page_size][head_dim] bf16 at element offset
 * (l * n_pages + p) * n_heads_kv * page_size * head_dim.
 * Logical cache position t lives in page page_table[t / page_size] at row
 * t % page_size.  page_table has ceil(capacity / page_size) entries.      */
typedef struct {
  sub_bf16* k;
  sub_bf16* v;
  const int32_t* page_table;   /* device */
  int32_t n_layers;
  int32_t n_heads_kv;
  int32_t head_dim;            /* 64 or 128 */
  int32_t page_size;           /* multiple of 16 */
  int32_t n_pages;
  int64_t capacity;            /* logical positions covered by page_table */
} sub_kv_cache;

/* Tree-masked GQA attention ("Low-Bit Shadow" report 6.3, SpecInfer: one
 * target pass verifies every tree node).  Query i (Q [n_q, Hq, d] bf16) reads
 *   - the committed keys at positions [0, n_prefix), and
 *   - the tree keys of its root path: for j in 0..depth[i], slot anc[i*anc_stride + j]
 *     stored at cache position tree_base + slot (anc lists root .. self).
 * anc == NULL means a chain: query i is slot i with path 0..i (a causal block,
 * as in prefill).  n_slots bounds the slot indices (max slot + 1, <= 16384).
 * O [n_q, Hq, d] bf16 = softmax(q K^T * softmax_scale) V, softmax in fp32.
 * Hq % Hkv == 0; head_dim 64 or 128.  Allocates nothing: key splits merge
 * inside one thread-block cluster. */
int32_t sub_tree_attn(const sub_bf16* Q, int32_t n_q, int32_t n_heads_q,
                      const sub_kv_cache* kv, int32_t layer, int64_t n_prefix, int64_t tree_base,
                      int32_t n_slots, const int32_t* anc, int32_t anc_stride,
                      const int32_t* depth, float softmax_scale, sub_bf16* O, void* stream);

/* ------------------------------------------------------------------------ */
/* Static token tree ("Low-Bit Shadow" report 6.3/6.4: deep, narrow, static,
 * k nodes per level, depth D).  Slot 0 is the root; level l in 1..D holds
 * slots 1+(l-1)k .. lk.  Device arrays sized for 1 + D*k slots;
 * anc is [1 + D*k][D + 1] (root .. self, -1 padded). */
typedef struct {
  int32_t* token;
  int32_t* parent;
  int32_t* depth;
  float* score;       /* cumulative sharpened log-probability */
  int32_t* anc;
  int32_t width;      /* k */
  int32_t max_depth;  /* D; anc row stride is D + 1 */
} sub_tree;

/* Expand level `level` (0 = root alone; else its k slots) into level+1.
 * logits: fp32 [k_prev, V] draft logits of the level's slots in slot order.
 * For each frontier node j: lp = z/T - logsumexp(z/T) (T = temperature,
 * "sharpened" draft probabilities: card, Approach; report 3.4), candidates =
 * its own top-k tokens (ties -> smaller id), score = S_j + lp; level+1 keeps
 * the global top-k (ties -> smaller parent slot, then smaller id) in
 * descending score order, writing token/parent/depth/score/anc.
 * 1 <= k <= 16, level < max_depth. */
int32_t sub_draft_expand(const float* logits, int64_t V, float temperature,
                         const sub_tree* tree, int32_t level, void* stream);

/* Verify + accept.  choice(u) = argmax_v logits[u, v] (mode 0, greedy) or
 * argmax_v logits[u, v]/T + g(seed, root_pos + depth(u) + 1, v) (mode 1,
 * Gumbel-max with Philox4x32-10 noise, Salmon et al. SC'11; counter
 * (v/4, position, 0, 0), key (seed lo, seed hi), word v%4, x = ((r>>9)+0.5)*2^-23,
 * g = -log(-log x)); ties -> smaller id.  Walk from the root to the child
 * whose token equals choice(current) while one exists ("Low-Bit Shadow"
 * report 6.2/6.3).  Writes accepted_slots[0..a), *n_accepted = a, *bonus_token
 * = choice(last), and choice[n_nodes] if choice != NULL. */
int32_t sub_verify_accept(const float* logits, const sub_tree* tree, int32_t n_nodes, int64_t V,
                          int32_t mode, float temperature, uint64_t seed, int64_t root_pos,
                          int32_t* accepted_slots, int32_t* n_accepted, int32_t* bonus_token,
                          int32_t* choice, void* stream);

/* sub_verify_accept without any device allocation: the same operation and
 * arguments, with its per-call scratch (partial argmax keys, the ticket
 * counter and, when choice == NULL, the choice array) taken from one fixed
 * array of device memory that the library holds for each device
 * (SUB_ACCEPT_STATIC_BYTES, 256 KB; every device that loads the library
 * keeps it until the process exits).  The paper has no counterpart: it is for
 * callers that cannot allocate device memory while they decode -- a runtime
 * that owns the device's memory through its own allocator and does not let
 * libraries call cudaMalloc or cudaMallocAsync, or a decode loop that must not
 * stall or fail on an allocation once it has started.  Requirement: n_nodes * chunks * 8 + 64 (+ n_nodes * 4 without
 * choice) <= SUB_ACCEPT_STATIC_BYTES, where chunks = the vocabulary chunks
 * per node (at most ceil(304 / n_nodes)); larger calls return SUB_EINVAL.
 * The first call on a device looks the array up (cudaGetSymbolAddress) and
 * must come before any stream capture on that device.  The array is shared:
 * calls on one device must be ordered (one stream, or joined by events);
 * two calls in flight at once race on it. */
#define SUB_ACCEPT_STATIC_BYTES (256 * 1024)
int32_t sub_verify_accept_static(const float* logits, const sub_tree* tree, int32_t n_nodes,
                                 int64_t V, int32_t mode, float temperature, uint64_t seed,
                                 int64_t root_pos, int32_t* accepted_slots, int32_t* n_accepted,
                                 int32_t* bonus_token, int32_t* choice, void* stream);

/* Commit the accepted path: for every layer and KV head, copy K,V of tree
 * slot accepted_slots[j-1] (at position root_pos + slot) to position
 * root_pos + j, j = 1..*n_accepted (read on the device).  The root stays at
 * root_pos.  Safe in place: all rows of a (layer, head) are read before any
 * is written. */
int32_t sub_kv_compact(const sub_kv_cache* kv, int64_t root_pos, const int32_t* accepted_slots,
                       const int32_t* n_accepted, int32_t max_accept, void* stream);

/* ------------------------------------------------------------------------ */
/* Model.  Layers [0, n_resident) keep bf16 weights on the device; layers
 * [n_resident, n_layers) are offloaded: their bf16 originals live in pinned
 * host memory and stream over the host link into a device staging ring for
 * every target pass, while their int4 substitutes (from sub_w4_pack) serve
 * the draft ("Low-Bit Shadow" report 2.1, 2.2 Step 4; card, measured
 * effects: asynchronous data transfer).  All weight matrices are
 * [out_features, in_features] row-major. */
typedef struct {
  const uint8_t* q;
  const sub_bf16* scale;
  const sub_bf16* zero;
  int32_t bits;   /* code bits: 2, 3 or 4 (0 means 4); see sub_wq_pack.  A layer's
                     q/k/v substitutes share one width, and so do gate and up;
                     draft forwards over more than 16 rows need 4 bits */
} sub_w4;

typedef struct {
  /* bf16 originals: device pointers (resident) or pinned host pointers (offloaded) */
  const sub_bf16 *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  const sub_bf16 *attn_norm, *ffn_norm;            /* device [hidden] */
  sub_w4 q4, k4, v4, o4, g4, u4, d4;                /* offloaded layers only */
} sub_layer_desc;

typedef struct {
  int32_t n_layers, hidden, n_heads_q, n_heads_kv, head_dim, ffn, vocab, n_resident;
  float rope_theta, rms_eps;
  const sub_bf16* embed;        /* [vocab, hidden]: device memory, or pinned host memory
                                   (cudaHostAlloc / cudaHostRegister), which the
                                   embedding kernel reads in place over the host
                                   link, one row per token (saves vocab*hidden*2
                                   bytes of device memory) */
  const sub_bf16* lm_head;      /* device [vocab, hidden] */
  const sub_bf16* final_norm;   /* device [hidden] */
  const sub_layer_desc* layers; /* host array [n_layers] */
  int32_t max_seq;              /* prompt + generated tokens the cache must hold */
  int32_t max_depth, max_width; /* largest tree the workspace is sized for */
  int32_t staging_layers;       /* device ring slots for streamed originals; 0 = all */
  int32_t max_prompt;           /* largest prompt (prefill rows) */
} sub_model_desc;

typedef struct sub_model sub_model;

int32_t sub_model_create(const sub_model_desc* desc, sub_model** out);
int32_t sub_model_destroy(sub_model* model);

/* Device memory the model holds (weights it allocated + workspace), bytes. */
int32_t sub_model_memory(const sub_model* model, int64_t* device_bytes);

/* One forward of the target (which = 0) or the draft (which = 1) over rows
 * that are tree slots [slot0, slot0 + n_rows) placed after a committed prefix of
 * n_prefix tokens: row r (slot s = slot0 + r) carries token tokens[r] at
 * position n_prefix + depth[r], reads positions [0, n_prefix) and the slots of
 * anc[r * anc_stride ...] (root .. self), and writes its K,V at position
 * n_prefix + s.  anc == NULL: chain (row r is slot slot0 + r, path 0..s).
 * logits: fp32 [n_rows, vocab], or NULL.  A prefill is a chain with
 * n_prefix = 0; a plain decode step is one row at slot 0. */
int32_t sub_model_forward(sub_model* model, int32_t which, const int32_t* tokens, int32_t n_rows,
                          int32_t slot0, const int32_t* depth, const int32_t* anc,
                          int32_t anc_stride, int64_t n_prefix, float* logits, void* stream);

/* The model's KV cache (for tests that inspect it). */
int32_t sub_model_kv(sub_model* model, sub_kv_cache* out);

typedef struct {
  int32_t depth;          /* D >= 0; 0 = plain target decoding */
  int32_t width;          /* k >= 1 */
  float draft_temp;       /* 0.2 in the pages */
  int32_t mode;           /* 0 greedy, 1 Gumbel-max sampling */
  float target_temp;
  uint64_t seed;
  int32_t use_graph;      /* capture one decode cycle as a CUDA graph */
  /* Adaptive depth ("Low-Bit Shadow" report 3.7 and 10.1 (3)): after each
   * level is added, drafting stops when the best cumulative sharpened
   * log-probability among its nodes is below stop_logp; the cycle then
   * verifies the tree with the levels drafted so far, and the accept walk
   * stops at the last of them.  Only a finite negative value turns this on:
   * 0 (a zero-filled config), -INFINITY and NaN draft all `depth` levels.
   * The decision is taken on the device in fp32.  In a captured cycle
   * (use_graph) the levels after the first are conditional graph nodes, so
   * a level not drafted launches nothing; without use_graph the host reads
   * the decision after every level (one synchronisation per level). */
  float stop_logp;
  /* Verify reuse of the draft's leading layers (layer and KV sharing, "Low-Bit
   * Shadow" report 4.1 point 2): layers [0, n_resident) are the target's own,
   * so the draft's residual stream after them is the target's for the same
   * node.  Nonzero: every tree node's leading part runs once, in the draft
   * (the deepest level's nodes get it right after their expansion), and the
   * verify starts at layer n_resident from it; the K/V of those layers are
   * the draft's.  The draft's kernels (M <= 16 GEMV) and the verify's (tiled
   * GEMM) round differently, so the verify logits move by that rounding
   * noise; the emitted tokens stay the target's up to near-ties. */
  int32_t verify_reuse;
} sub_decode_cfg;

typedef struct {
  int64_t cycles;         /* verify passes after the prefill */
  int64_t emitted;        /* tokens generated (= n_new) */
  double tau;             /* tokens per verify pass, counting the bonus */
  double t_prefill_ms;
  double t_decode_ms;
  int64_t accept_hist[65];/* cycles that accepted a tokens, a <= 64 */
  /* Per-phase device time summed over the cycles (CUDA events on the
   * compute stream; -1 where the device could not time them):
   *   t_draft_ms   the D draft levels (forwards + expansions),
   *   t_verify_ms  the target pass over the tree (it waits for the streamed
   *                originals of offloaded layers),
   *   t_copy_unhidden_ms  the part of the verify spent waiting for those
   *                copies: per offloaded layer, how long after the compute
   *                stream reached the layer its copy finished (0 if before).
   * t_draft_ms / t_verify_ms is the draft-to-target cost term
   * D * t_draft_level / t_target of the speedup's denominator ("Low-Bit
   * Shadow" report 7.1). */
  double t_draft_ms;
  double t_verify_ms;
  double t_copy_unhidden_ms;
  /* emitted tokens whose best and runner-up choice scores (logits, or
   * logits / T + Gumbel noise) differed by less than 1e-2 on the device: the
   * positions where a rounding difference could pick another token */
  int64_t near_tie_events;
  /* draft levels run over all cycles (cycles * depth without adaptive depth) */
  int64_t drafted_levels;
  /* device time from each cycle's start to the last offloaded original
   * landing in the staging ring, summed over cycles (0 without offloaded
   * layers): streamed bytes / t_copy_ms is the host link rate the cycles got */
  double t_copy_ms;
} sub_stats;

/* Step-wise decoding (the pieces sub_generate is made of).
 * sub_prefill: reset the decode state, run the target over the prompt
 *   (streaming offloaded layers), and emit the first token.  Enqueued on
 *   `stream`; nothing is read back.
 * sub_decode_cycles: enqueue n_cycles draft/verify/accept/compact cycles on
 *   `stream` without any host synchronisation (as CUDA-graph replays when
 *   cfg->use_graph; the graph is captured on first use per configuration).
 *   Emitted tokens accumulate on the device; the caller must keep
 *   n_prompt + emitted + depth + 1 <= max_seq.
 * sub_decode_read: synchronise the model's stream, then copy the emitted
 *   stream (int32 [min(n, emitted)]) to out_host and return the count of
 *   emitted tokens and of cycles run since the prefill. */
int32_t sub_prefill(sub_model* model, const int32_t* prompt_host, int32_t n_prompt,
                    const sub_decode_cfg* cfg, void* stream);
int32_t sub_decode_cycles(sub_model* model, const sub_decode_cfg* cfg, int32_t n_cycles,
                          void* stream);
int32_t sub_decode_read(sub_model* model, int32_t* out_host, int32_t n, int32_t* emitted,
                        int64_t* cycles);

/* Per-cycle facts of the captured graph for configuration cfg (captures it
 * if needed): kernels launched per cycle and host->device bytes streamed per
 * cycle (the offloaded originals). */
int32_t sub_cycle_info(sub_model* model, const sub_decode_cfg* cfg, int64_t* kernels_per_cycle,
                       int64_t* h2d_bytes_per_cycle);

/* Generate n_new tokens after prompt_host (int32 [n_prompt], host) into
 * out_tokens_host (int32 [n_new], host): prefill, then draft/verify/accept
 * cycles until n_new tokens are emitted (the first comes from the prefill;
 * the last cycle is truncated).  Synchronous.  stats may be NULL.
 * Returns SUB_ETIMEOUT (tokens and stats still written) when a bounded
 * pipeline wait ran out during the call: the tokens are then not to be
 * trusted.  sub_decode_read does the same check since the last prefill. */
int32_t sub_generate(sub_model* model, const int32_t* prompt_host, int32_t n_prompt,
                     int32_t n_new, const sub_decode_cfg* cfg, int32_t* out_tokens_host,
                     sub_stats* stats);

#ifdef __cplusplus
}
#endif
#endif /* SUB_API_H */
