// Static draft tree kernels: expansion of one level from sharpened draft
// probabilities, the target's choice per node with the accept walk, and the
// compaction of the accepted path in the shared KV cache.
//
// Expansion ("SubSpec: Using the Target Model's Own Low-Bit Shadow as Its
// Draft Model", 6.3/6.4: deep, narrow, static tree of width k; "Speculate Deep
// and Accurate" card, Approach: draft probabilities sharpened with T = 0.2):
// per frontier node j, lp = z/T - logsumexp(z/T); its own top-k tokens are
// the candidates (ties -> smaller id); score = S_j + lp; the next level keeps
// the global top-k (ties -> smaller parent slot, then smaller id).
//
// Accept (report 6.2 Leviathan et al., 6.3 SpecInfer): choice(u) is the
// target's argmax (greedy) or Gumbel-max sample with noise keyed by (seed,
// position); walk from the root into the child whose token equals the choice.
//
// Both reductions over the vocabulary split it into chunks over CTAs and
// finish in the last CTA to arrive (a ticket counter the kernel resets), in a
// fixed order, so results are deterministic and a single launch suffices.
#include "tree.cuh"

namespace sub {

// ------------------------------------------------------------ helpers --
template <int N>
__device__ __forceinline__ void topn_insert(unsigned long long (&top)[N], unsigned long long key) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (key > top[i]) {
      const unsigned long long t = top[i];
      top[i] = key;
      key = t;
    }
  }
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Block-wide max of a 64-bit key (256 threads); all threads get the result.
__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  unsigned long long r = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = s_red[i] > r ? s_red[i] : r;
  return r;
}

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  if (m2 > m) { s = s * expf(m - m2) + s2; m = m2; }
  else s += s2 * expf(m2 - m);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}
__device__ __forceinline__ float gumbel_of(uint32_t r) {
  const float x = ((float)(r >> 9) + 0.5f) * 1.1920928955078125e-07f;   // 2^-23, exact
  return -logf(-logf(x));
}

// ------------------------------------------------------------- expand --
constexpr int EXP_THREADS = 256;

size_t expand_scratch_bytes(int k_prev, int n_chunks, int width) {
  const size_t parts = (size_t)k_prev * n_chunks;
  return parts * MAX_WIDTH * 8 + parts * 8 + 64;
}
int expand_pick_chunks(int k_prev, int64_t V) {
  int c = (int)((2 * 152 + k_prev - 1) / k_prev);
  c = std::min<int64_t>(c, (V + 1023) / 1024);
  return std::max(1, std::min(c, 64));
}

template <int MAXK>
__global__ void __launch_bounds__(EXP_THREADS) expand_kernel(ExpandArgs a) {
  __shared__ unsigned long long s_red[EXP_THREADS / 32];
  __shared__ float s_m[EXP_THREADS / 32], s_s[EXP_THREADS / 32];
  __shared__ unsigned int s_last;
  pdl_wait();
  pdl_trigger();
  const int k = a.tree.width;
  const int j = blockIdx.y, c = blockIdx.x;
  const int64_t V = a.V;
  const int64_t cs = (V + a.n_chunks - 1) / a.n_chunks;
  const int64_t lo = c * cs, hi = min(V, lo + cs);
  const float* z = a.logits + (int64_t)j * V;

  unsigned long long top[MAXK];
#pragma unroll
  for (int i = 0; i < MAXK; ++i) top[i] = 0ull;
  float m = -INFINITY, s = 0.f;
  for (int64_t v = lo + threadIdx.x; v < hi; v += EXP_THREADS) {
    const float zv = z[v];
    const float zt = __fdiv_rn(zv, a.temp);
    if (zt > m) { s = (m == -INFINITY ? 0.f : s * expf(m - zt)) + 1.f; m = zt; }
    else s += expf(zt - m);
    const unsigned long long key = rank_key(zv, (uint32_t)v);
    if (key > top[MAXK - 1]) topn_insert(top, key);
  }
  // block merge of (m, s) in warp then warp-index order
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { s_m[warp] = m; s_s[warp] = s; }
  // block top-k: k rounds of block argmax; the winner shifts its sorted list
  const size_t part = (size_t)j * a.n_chunks + c;
  for (int r = 0; r < k; ++r) {
    const unsigned long long best = block_max_u64(top[0], s_red);
    if (top[0] == best && best != 0ull) {
#pragma unroll
      for (int i = 0; i < MAXK - 1; ++i) top[i] = top[i + 1];
      top[MAXK - 1] = 0ull;
    }
    if (threadIdx.x == 0) a.part_key[part * MAX_WIDTH + r] = best;
  }
  if (threadIdx.x == 0) {
    float bm = -INFINITY, bs = 0.f;
    for (int w = 0; w < EXP_THREADS / 32; ++w) lse_merge(bm, bs, s_m[w], s_s[w]);
    a.part_max[part] = bm;
    a.part_sum[part] = bs;
    __threadfence();
    const unsigned int total = gridDim.x * gridDim.y;
    s_last = (atomicAdd(a.counter, 1u) == total - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---------------- last CTA: per-row lse and top-k, then the global top-k
  __shared__ float s_lse[MAX_WIDTH];
  __shared__ unsigned long long s_cand[MAX_WIDTH * MAX_WIDTH];   // [row][i] token keys
  __shared__ unsigned long long s_glob[MAX_WIDTH * MAX_WIDTH];   // score keys
  const int kp = a.k_prev;
  // every CTA's partial results into shared memory first, eight loads in
  // flight per thread (read one at a time they put a round trip per chunk
  // on the launch's tail)
  const int n_part = kp * a.n_chunks;
  extern __shared__ unsigned long long s_dyn[];
  unsigned long long* const s_key = s_dyn;                        // [part][k]
  float* const s_pm = reinterpret_cast<float*>(s_key + (size_t)n_part * k);
  float* const s_ps = s_pm + n_part;
  for (int i0 = threadIdx.x; i0 < n_part * k; i0 += 8 * EXP_THREADS) {
    unsigned long long v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * EXP_THREADS;
      v[u] = i < n_part * k ? __ldcg(a.part_key + (size_t)(i / k) * MAX_WIDTH + i % k) : 0ull;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (i0 + u * EXP_THREADS < n_part * k) s_key[i0 + u * EXP_THREADS] = v[u];
  }
  for (int i0 = threadIdx.x; i0 < n_part; i0 += 2 * EXP_THREADS) {
    const int i1 = i0 + EXP_THREADS;
    const float m0 = __ldcg(a.part_max + i0), q0 = __ldcg(a.part_sum + i0);
    const float m1 = i1 < n_part ? __ldcg(a.part_max + i1) : 0.f;
    const float q1 = i1 < n_part ? __ldcg(a.part_sum + i1) : 0.f;
    s_pm[i0] = m0;
    s_ps[i0] = q0;
    if (i1 < n_part) {
      s_pm[i1] = m1;
      s_ps[i1] = q1;
    }
  }
  __syncthreads();
  if (threadIdx.x < kp) {
    float bm = -INFINITY, bs = 0.f;
    for (int cc = 0; cc < a.n_chunks; ++cc) {
      const int p = threadIdx.x * a.n_chunks + cc;
      lse_merge(bm, bs, s_pm[p], s_ps[p]);
    }
    s_lse[threadIdx.x] = bm + logf(bs);
  }
  // per-row top-k over n_chunks * k candidates: warp w handles rows w, w+8, ...
  for (int row = warp; row < kp; row += EXP_THREADS / 32) {
    const int nc = a.n_chunks * k;
    for (int r = 0; r < k; ++r) {
      unsigned long long best = 0ull;
      for (int i = lane; i < nc; i += 32) {
        const unsigned long long key = s_key[(size_t)row * nc + i];
        bool taken = false;
        for (int q = 0; q < r; ++q) taken |= (s_cand[row * MAX_WIDTH + q] == key);
        if (!taken && key > best) best = key;
      }
      best = warp_max_u64(best);
      if (lane == 0) s_cand[row * MAX_WIDTH + r] = best;
      __syncwarp();
    }
  }
  __syncthreads();
  // candidate scores; frontier slots of this level
  const int level = a.level;
  const int slot_base = level == 0 ? 0 : 1 + (level - 1) * k;
  const int n_cand = kp * k;
  for (int i = threadIdx.x; i < n_cand; i += EXP_THREADS) {
    const int row = i / k, r = i % k;
    const unsigned long long key = s_cand[row * MAX_WIDTH + r];
    unsigned long long gk = 0ull;
    if (key != 0ull) {
      const uint32_t v = rank_idx(key);
      const float zt = __fdiv_rn(a.logits[(int64_t)row * V + v], a.temp);
      const int pslot = slot_base + row;
      const float score = a.tree.score[pslot] + (zt - s_lse[row]);
      // ties: smaller parent slot, then smaller token id (slot < 2^12, id < 2^20)
      gk = ((unsigned long long)float_key(score) << 32) |
           (unsigned long long)(0xffffffffu - (((uint32_t)pslot << 20) | v));
    }
    s_glob[i] = gk;
  }
  __syncthreads();
  if (warp == 0) {
    const int out0 = 1 + level * k;
    const int D = a.tree.max_depth;
    for (int r = 0; r < k; ++r) {
      unsigned long long best = 0ull;
      int bi = -1;
      for (int i = lane; i < n_cand; i += 32)
        if (s_glob[i] > best) { best = s_glob[i]; bi = i; }
      const unsigned long long wbest = warp_max_u64(best);
      if (best == wbest && bi >= 0 && best != 0ull) s_glob[bi] = 0ull;   // unique keys
      __syncwarp();
      if (lane == 0) {
        const uint32_t low = 0xffffffffu - (uint32_t)(wbest & 0xffffffffull);
        const int pslot = (int)(low >> 20);
        const int v = (int)(low & 0xfffffu);
        const int slot = out0 + r;
        a.tree.token[slot] = v;
        a.tree.parent[slot] = pslot;
        a.tree.depth[slot] = level + 1;
        a.tree.score[slot] = key_float((uint32_t)(wbest >> 32));
      }
      __syncwarp();
    }
    // ancestor lists: parent's list + self
    for (int i = lane; i < k * (D + 1); i += 32) {
      const int r = i / (D + 1), jj = i % (D + 1);
      const int slot = out0 + r;
      const int pslot = a.tree.parent[slot];
      int val = -1;
      if (jj <= level) val = a.tree.anc[(size_t)pslot * (D + 1) + jj];
      else if (jj == level + 1) val = slot;
      a.tree.anc[(size_t)slot * (D + 1) + jj] = val;
    }
  }
  if (threadIdx.x == 0) *a.counter = 0u;
}

int32_t launch_expand(const ExpandArgs& a, cudaStream_t st) {
  const int k = a.tree.width;
  SUB_CHECK_ARG(k >= 1 && k <= MAX_WIDTH, "expand: width must be in [1, 16]");
  SUB_CHECK_ARG(a.level >= 0 && a.level < a.tree.max_depth, "expand: level out of range");
  SUB_CHECK_ARG(a.V >= k && a.V <= (1 << 20), "expand: V must be in [k, 2^20]");
  SUB_CHECK_ARG(1 + (int64_t)a.tree.max_depth * k < 4096, "expand: tree too large");
  SUB_CHECK_ARG(a.temp > 0.f, "expand: temperature must be positive");
  SUB_CHECK_ARG(a.n_chunks >= 1 && a.k_prev >= 1 && a.k_prev <= MAX_WIDTH, "expand: bad split");
  dim3 grid(a.n_chunks, a.k_prev);
  // the last CTA stages every partial: keys [parts][k], then max and sum per part
  const size_t smem = (size_t)a.n_chunks * a.k_prev * (k * 8 + 8);
  SUB_CHECK_ARG(smem <= 43 * 1024, "expand: too many chunks for the staging buffer");
  if (k <= 8) SUB_CUDA_TRY(launch_k(expand_kernel<8>, grid, dim3(EXP_THREADS), smem, st, a));
  else SUB_CUDA_TRY(launch_k(expand_kernel<16>, grid, dim3(EXP_THREADS), smem, st, a));
  return SUB_OK;
}

// ------------------------------------------------------------- accept --
constexpr int ACC_THREADS = 256;

size_t accept_scratch_bytes(int n_nodes, int n_chunks) {
  return (size_t)n_nodes * n_chunks * 8 + 64;
}
int accept_pick_chunks(int n_nodes, int64_t V) {
  int c = (int)((2 * 152 + n_nodes - 1) / n_nodes);
  c = std::min<int64_t>(c, (V + 4095) / 4096);
  return std::max(1, std::min(c, 64));
}

__global__ void __launch_bounds__(ACC_THREADS) accept_kernel(AcceptArgs a) {
  __shared__ unsigned long long s_red[ACC_THREADS / 32];
  __shared__ unsigned int s_last;
  pdl_wait();
  pdl_trigger();
  const int u = blockIdx.y, c = blockIdx.x;
  const int64_t V = a.V;
  // chunks of whole 4-token Philox blocks
  const int64_t blocks4 = (V + 3) / 4;
  const int64_t cb = (blocks4 + a.n_chunks - 1) / a.n_chunks;
  const int64_t b_lo = c * cb, b_hi = min(blocks4, b_lo + cb);
  const float* z = a.logits + (int64_t)u * V;
  const int64_t root_pos = a.root_pos_dev ? (int64_t)*a.root_pos_dev : a.root_pos;
  const uint32_t pos = (uint32_t)(root_pos + a.tree.depth[u] + 1);
  const uint32_t k0 = (uint32_t)(a.seed & 0xffffffffull), k1 = (uint32_t)(a.seed >> 32);
  unsigned long long best = 0ull, second = 0ull;
  for (int64_t b = b_lo + threadIdx.x; b < b_hi; b += ACC_THREADS) {
    uint4 r = make_uint4(0, 0, 0, 0);
    if (a.mode == 1) r = philox4x32_10(make_uint4((uint32_t)b, pos, 0u, 0u), k0, k1);
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t v = b * 4 + i;
      if (v >= V) break;
      float sc = z[v];
      if (a.mode == 1) sc = __fdiv_rn(sc, a.temp) + gumbel_of(rw[i]);
      const unsigned long long key = rank_key(sc, (uint32_t)v);
      if (key > best) {
        second = best;
        best = key;
      } else if (key > second) {
        second = key;
      }
    }
  }
  const unsigned long long mine = best;
  best = block_max_u64(best, s_red);
  if (a.near_ties) {
    // the chunk's runner-up: the best key of the thread that held the winner
    // is replaced by that thread's second
    second = block_max_u64(mine == best ? second : mine, s_red);
    if (threadIdx.x == 0) a.part_key2[(size_t)u * a.n_chunks + c] = second;
  }
  if (threadIdx.x == 0) {
    a.part_key[(size_t)u * a.n_chunks + c] = best;
    __threadfence();
    s_last = (atomicAdd(a.counter, 1u) == gridDim.x * gridDim.y - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA: choice per node, then the walk
  for (int n = threadIdx.x; n < a.n_nodes; n += ACC_THREADS) {
    unsigned long long b2 = 0ull;
    for (int cc = 0; cc < a.n_chunks; ++cc) {
      const unsigned long long kk = a.part_key[(size_t)n * a.n_chunks + cc];
      b2 = kk > b2 ? kk : b2;
    }
    a.choice[n] = (int32_t)rank_idx(b2);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int k = a.tree.width;
    int cur = 0, n_acc = 0;
    const int dlim = a.depth_limit ? *a.depth_limit : 0x7fffffff;
    while (true) {
      const int d = a.tree.depth[cur];
      if (d >= dlim) break;   // no drafted level below this node
      const int lo = 1 + d * k, hi = min(a.n_nodes, lo + k);
      int next = -1;
      for (int s = lo; s < hi; ++s)
        if (a.tree.parent[s] == cur && a.tree.token[s] == a.choice[cur]) { next = s; break; }
      if (next < 0) break;
      a.accepted[n_acc++] = next;
      cur = next;
    }
    const int bonus = a.choice[cur];
    *a.n_accepted = n_acc;
    *a.bonus = bonus;
    if (a.out_tokens) {
      const int e = *a.state_emitted;
      for (int i = 0; i < n_acc; ++i) a.out_tokens[e + i] = a.tree.token[a.accepted[i]];
      a.out_tokens[e + n_acc] = bonus;
      *a.state_emitted = e + n_acc + 1;
    }
    if (a.hist) a.hist[n_acc] += 1;
    if (a.near_ties) {
      // path nodes root, accepted[0..n_acc): their choices are the emitted tokens
      int ties = 0;
      for (int i = 0; i <= n_acc; ++i) {
        const int node = i == 0 ? 0 : a.accepted[i - 1];
        unsigned long long k1 = 0ull, k2 = 0ull;
        for (int cc = 0; cc < a.n_chunks; ++cc) {
          const unsigned long long b1 = a.part_key[(size_t)node * a.n_chunks + cc];
          const unsigned long long b2 = a.part_key2[(size_t)node * a.n_chunks + cc];
          if (b1 > k1) {
            k2 = k1 > b2 ? k1 : b2;
            k1 = b1;
          } else {
            k2 = b1 > k2 ? b1 : k2;
          }
        }
        if (k2 != 0ull &&
            key_float((uint32_t)(k1 >> 32)) - key_float((uint32_t)(k2 >> 32)) < a.tie_gap)
          ++ties;
      }
      *a.near_ties += ties;
    }
    *a.counter = 0u;
  }
}

int32_t launch_accept(const AcceptArgs& a, cudaStream_t st) {
  SUB_CHECK_ARG(a.n_nodes >= 1 && a.V >= 1, "accept: empty input");
  SUB_CHECK_ARG(a.mode == 0 || a.mode == 1, "accept: mode must be 0 or 1");
  SUB_CHECK_ARG(a.mode == 0 || a.temp > 0.f, "accept: temperature must be positive");
  SUB_CHECK_ARG(a.V < (1ll << 32), "accept: V too large");
  SUB_CHECK_ARG(a.choice != nullptr, "accept: choice buffer required");
  dim3 grid(a.n_chunks, a.n_nodes);
  SUB_CUDA_TRY(launch_k(accept_kernel, grid, dim3(ACC_THREADS), 0, st, a));
  return SUB_OK;
}

// ------------------------------------------------------------ compact --
// One CTA per (layer, KV head): read every accepted row, then write them, so
// a destination that is also a later source cannot be clobbered.
__global__ void compact_kernel(CompactArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  const int layer = blockIdx.x, h = blockIdx.y;
  const int n = min(*a.n_accepted, a.max_accept);
  if (n <= 0) return;
  const int64_t root = a.root_pos_dev ? (int64_t)*a.root_pos_dev : a.root_pos;
  const int D = a.head_dim, CH = D / 8;
  const size_t head_stride = (size_t)a.page_size * D;
  const size_t page_stride = (size_t)a.n_heads_kv * head_stride;
  const size_t layer_off = (size_t)layer * a.n_pages * page_stride;
  auto addr = [&](int64_t p) {
    return layer_off + (size_t)a.page_table[p / a.page_size] * page_stride +
           (size_t)h * head_stride + (size_t)(p % a.page_size) * D;
  };
  uint4* sk = reinterpret_cast<uint4*>(smem);
  uint4* sv = sk + (size_t)a.max_accept * CH;
  for (int i = threadIdx.x; i < n * CH; i += blockDim.x) {
    const int j = i / CH, c = i % CH;
    const size_t src = addr(root + a.accepted[j]) + c * 8;
    sk[i] = *reinterpret_cast<const uint4*>(a.k + src);
    sv[i] = *reinterpret_cast<const uint4*>(a.v + src);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n * CH; i += blockDim.x) {
    const int j = i / CH, c = i % CH;
    const size_t dst = addr(root + 1 + j) + c * 8;
    *reinterpret_cast<uint4*>(a.k + dst) = sk[i];
    *reinterpret_cast<uint4*>(a.v + dst) = sv[i];
  }
}

int32_t launch_compact(const CompactArgs& a, cudaStream_t st) {
  SUB_CHECK_ARG(a.head_dim % 8 == 0 && a.head_dim <= 256, "compact: bad head_dim");
  SUB_CHECK_ARG(a.max_accept >= 0 && a.max_accept <= 256, "compact: max_accept out of range");
  if (a.max_accept == 0) return SUB_OK;
  const int smem = 2 * a.max_accept * a.head_dim * 2;
  dim3 grid(a.n_layers, a.n_heads_kv);
  SUB_CUDA_TRY(launch_k(compact_kernel, grid, dim3(128), smem, st, a));
  return SUB_OK;
}

}  // namespace sub
