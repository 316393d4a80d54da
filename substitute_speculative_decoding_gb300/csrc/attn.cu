// Tree-masked GQA attention over the paged shared KV cache.
//
// Tree verification scores every node of the draft tree in one target pass:
// node u reads the committed prefix plus the keys of its own root path
// ("SubSpec: Using the Target Model's Own Low-Bit Shadow as Its Draft Model",
// 6.3 SpecInfer); the draft reads the same shared cache (report 4.1 point 2).
//
// Key index space of one call: j < n_prefix is cache position j (visible to
// every query); j = n_prefix + s is tree slot s at position tree_base + s,
// visible to query i when s is on i's root path (a per-query bitmap built in
// shared memory from the ancestor lists; a chain when no lists are given).
//
// Rows are (query, head-in-group) pairs of one KV head, so the Hq/Hkv query
// heads that share a KV head read each K/V tile once.  A CTA of four warps
// owns 64 rows; S = Q K^T and O += P V run on mma.sync m16n8k16 with fp32
// accumulators and an online softmax in fp32 (FlashAttention-2 style); P
// enters P V as a bf16 pair hi + lo, which keeps it to ~2^-17.  Keys
// may be split over up to 16 CTAs (grid.z) that form one thread-block cluster;
// their partial (max, sum, O) are merged in split order through distributed
// shared memory, so no global scratch and no second launch are needed.  Long
// key ranges with few row blocks take 32 splits: four clusters of 8, each
// merged as above, whose partials meet in a small global scratch and are
// folded, in cluster order, by the last CTA of each row slice to arrive.
#include <mutex>
#include <cooperative_groups.h>
#include "attn_core.cuh"

namespace sub {

template <int D>
__global__ void __launch_bounds__(THREADS) tree_attn_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  float o[D / 8][4], m_run[2], l_run[2];
  attn_main<D>(a, blockIdx.y, blockIdx.x * ROWS, blockIdx.z, gridDim.z, smem,
               [] { __syncthreads(); }, o, m_run, l_run);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int wrow = warp * 16;
  const int kvh = blockIdx.y;
  const int G = a.n_heads_q / a.n_heads_kv;
  const int n_rows = a.n_q * G;
  const int row0 = blockIdx.x * ROWS;
  uint8_t* sK = smem + ROWS * D * 2;

  pdl_trigger();
  // ---- write out ----
  if (gridDim.z == 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gr = row0 + wrow + g + 8 * h;
      if (gr >= n_rows) continue;
      const int q = gr / G, hh = gr % G;
      const size_t orow = (size_t)q * a.n_heads_q + kvh * G + hh;   // row of [n_q*Hq]
      const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const int c = i * 8 + 2 * tig;
        *reinterpret_cast<uint32_t*>(a.O + orow * D + c) =
            pack_bf16x2(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
      }
    }
    return;
  }
  // Key splits form one thread-block cluster: each CTA parks its partial
  // (max, sum, unnormalised O) in its own shared memory, and after a cluster
  // barrier every CTA merges a slice of the rows by reading its peers' shared
  // memory (distributed shared memory), in split order: the peers' maxima and
  // sums once per (row, split) into local memory, then one round of their
  // partial outputs, four columns per thread.
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int PLD = D + 4;
  float* sO = reinterpret_cast<float*>(sK);            // [ROWS][PLD], reuses the K/V tiles
  float* sM = sO + ROWS * PLD;                          // [ROWS]
  float* sL = sM + ROWS;                                // [ROWS]
  float* const sMl = sL + ROWS;                         // [rows_per][S] peer maxima
  float* const sWl = sMl + ROWS * ATTN_MAX_SPLIT;       // [rows_per][S] merge weights
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = wrow + g + 8 * h;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2*>(sO + r * PLD + i * 8 + 2 * tig) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
    if (tig == 0) {
      sM[r] = m_run[h];
      sL[r] = l_run[h];
    }
  }
  cluster.sync();
  const int S = (int)cluster.dim_blocks().z;   // splits of this cluster
  const int C = (int)gridDim.z / S;            // clusters of this row block (2-level merge if > 1)
  const int rank = (int)cluster.block_rank();
  const int rows_per = (ROWS + S - 1) / S;
  const int r_lo = rank * rows_per, r_hi = min(ROWS, r_lo + rows_per);
  const int n_ms = (r_hi - r_lo) * S;
  const bool act = tid < n_ms;
  const int mi = act ? tid / S : 0, ms2 = act ? tid % S : 0;
  float l_peer = 0.f, w_peer = 0.f;
  if (act) {
    sMl[mi * S + ms2] = cluster.map_shared_rank(sM, ms2)[r_lo + mi];
    l_peer = cluster.map_shared_rank(sL, ms2)[r_lo + mi];
  }
  __syncthreads();
  if (act) {
    float mx = -INFINITY;
    for (int t2 = 0; t2 < S; ++t2) mx = fmaxf(mx, sMl[mi * S + t2]);
    const float m2 = sMl[mi * S + ms2];
    w_peer = (m2 == -INFINITY) ? 0.f : exp2f(m2 - mx);
    sWl[mi * S + ms2] = w_peer * l_peer;   // this split's share of the denominator
  }
  __syncthreads();
  float den = 0.f;
  if (act)
    for (int t2 = 0; t2 < S; ++t2) den += sWl[mi * S + t2];   // in split order
  __syncthreads();
  // one cluster: normalised weights; several: this cluster's unnormalised
  // partial, its max and its denominator go to the cross-cluster scratch
  const size_t blk = (size_t)blockIdx.x * gridDim.y + blockIdx.y;
  const int c_idx = (int)blockIdx.z / S;
  if (act) sWl[mi * S + ms2] = C > 1 ? w_peer : w_peer * (den > 0.f ? 1.f / den : 0.f);
  if (C > 1 && act && ms2 == 0) {
    float mx = -INFINITY;
    for (int t2 = 0; t2 < S; ++t2) mx = fmaxf(mx, sMl[mi * S + t2]);
    const size_t xr = (blk * C + c_idx) * ROWS + r_lo + mi;
    a.xm[xr] = mx;
    a.xl[xr] = den;
  }
  __syncthreads();
  for (int idx = tid; idx < (r_hi - r_lo) * (D / 4); idx += THREADS) {
    const int i = idx / (D / 4), c = (idx % (D / 4)) * 4;
    const int r = r_lo + i;
    const int gr = row0 + r;
    if (gr >= n_rows) continue;
    float4 pv[ATTN_MAX_SPLIT];
#pragma unroll
    for (int s2 = 0; s2 < ATTN_MAX_SPLIT; ++s2)
      pv[s2] = s2 < S ? *reinterpret_cast<const float4*>(cluster.map_shared_rank(sO, s2) + r * PLD + c)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < ATTN_MAX_SPLIT; ++s2) {
      if (s2 < S) {
        const float w = sWl[i * S + s2];
        v0 = fmaf(w, pv[s2].x, v0);
        v1 = fmaf(w, pv[s2].y, v1);
        v2 = fmaf(w, pv[s2].z, v2);
        v3 = fmaf(w, pv[s2].w, v3);
      }
    }
    if (C > 1) {
      __stcg(reinterpret_cast<float4*>(a.xpart + ((blk * C + c_idx) * ROWS + r) * D + c),
             make_float4(v0, v1, v2, v3));
      continue;
    }
    const int q = gr / G, hh = gr % G;
    const size_t orow = (size_t)q * a.n_heads_q + kvh * G + hh;
    *reinterpret_cast<uint2*>(a.O + orow * D + c) = make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
  }
  if (C > 1) {
    // the rank-r CTAs of the C clusters hold the same rows: the last of them
    // to arrive merges the clusters' partials, in cluster order
    __shared__ unsigned int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.xcnt + blk * S + rank, 1u) == (unsigned)C - 1 ? 1u : 0u;
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int idx = tid; idx < (r_hi - r_lo) * (D / 4); idx += THREADS) {
        const int i = idx / (D / 4), c = (idx % (D / 4)) * 4;
        const int r = r_lo + i;
        const int gr = row0 + r;
        if (gr >= n_rows) continue;
        float M = -INFINITY;
        for (int cc = 0; cc < C; ++cc) M = fmaxf(M, __ldcg(a.xm + (blk * C + cc) * ROWS + r));
        float L = 0.f, v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
        for (int cc = 0; cc < C; ++cc) {
          const size_t xr = (blk * C + cc) * ROWS + r;
          const float mc = __ldcg(a.xm + xr);
          const float wc = mc == -INFINITY ? 0.f : exp2f(mc - M);
          const float4 p = __ldcg(reinterpret_cast<const float4*>(a.xpart + xr * D + c));
          L = fmaf(wc, __ldcg(a.xl + xr), L);
          v0 = fmaf(wc, p.x, v0);
          v1 = fmaf(wc, p.y, v1);
          v2 = fmaf(wc, p.z, v2);
          v3 = fmaf(wc, p.w, v3);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const int q = gr / G, hh = gr % G;
        const size_t orow = (size_t)q * a.n_heads_q + kvh * G + hh;
        *reinterpret_cast<uint2*>(a.O + orow * D + c) =
            make_uint2(pack_bf16x2(v0 * inv, v1 * inv), pack_bf16x2(v2 * inv, v3 * inv));
      }
      if (tid == 0) a.xcnt[blk * S + rank] = 0u;   // ready for the next launch
    }
  }
  cluster.sync();   // peers may still be reading this CTA's shared memory
}

int attn_smem_bytes(const AttnArgs& a) {
  const int d = a.head_dim;
  const int G = a.n_heads_q / a.n_heads_kv;
  const int nq = ROWS / G + 2;
  const int words = (a.n_slots + 31) / 32;
  return ROWS * d * 2 + 4 * KT * d * 2 + (a.anc ? nq * words * 4 : 0);
}
static_assert(ROWS * (128 + 4) * 4 + 2 * ROWS * 4 + 2 * ROWS * ATTN_MAX_SPLIT * 4 <= 4 * KT * 128 * 2,
              "the cluster merge buffers must fit in the K/V tiles (head_dim 128)");
static_assert(ROWS * (64 + 4) * 4 + 2 * ROWS * 4 + 2 * ROWS * ATTN_MAX_SPLIT * 4 <= 4 * KT * 64 * 2,
              "the cluster merge buffers must fit in the K/V tiles (head_dim 64)");

static int g_max_split = 8;   // largest cluster the device runs (set by attn_init)

int attn_pick_splits(const AttnArgs& a, int n_keys_hint, bool two_level) {
  if (attn_init() != SUB_OK) return 1;
  const int G = a.n_heads_q / a.n_heads_kv;
  const int blocks = (a.n_q * G + ROWS - 1) / ROWS * a.n_heads_kv;
  const int tiles = (n_keys_hint + KT - 1) / KT;
  int s = (2 * 152 + blocks - 1) / blocks;
  // past one cluster: four clusters of 8 per row block when the launch still
  // fits two CTAs per SM and every split keeps four key tiles or more (at
  // fewer keys the cross-cluster merge costs more than the added CTAs gain)
  if (two_level && g_max_split == 16 && s >= 32 && tiles >= 128) return 32;
  s = std::max(1, std::min(s, std::min(tiles, g_max_split)));
  return s;
}

size_t attn_xpart_floats(const AttnArgs& a, int n_split) {
  if (n_split <= ATTN_MAX_SPLIT) return 0;
  const int G = a.n_heads_q / a.n_heads_kv;
  const size_t blocks = (size_t)(a.n_q * G + ROWS - 1) / ROWS * a.n_heads_kv;
  const size_t C = (size_t)n_split / ATTN_XCLUSTER;
  return blocks * C * ROWS * (a.head_dim + 2);
}
size_t attn_xcnt_count(const AttnArgs& a, int n_split) {
  if (n_split <= ATTN_MAX_SPLIT) return 0;
  const int G = a.n_heads_q / a.n_heads_kv;
  return (size_t)(a.n_q * G + ROWS - 1) / ROWS * a.n_heads_kv * ATTN_XCLUSTER;
}

// Opt the kernels into the largest dynamic shared memory and into 16-CTA
// clusters once per process (before any stream capture: model creation
// calls this), and find whether the device runs clusters of 16.
int32_t attn_init() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const void* ks[2] = {(const void*)tree_attn_kernel<128>, (const void*)tree_attn_kernel<64>};
    for (const void* k : ks) {
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, ATTN_MAX_SMEM);
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    if (err != cudaSuccess) return;
    // can a 16-CTA cluster of the largest draft-shaped launch be resident?
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 16);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = ROWS * 128 * 2 + 4 * KT * 128 * 2 + 4096;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 16;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tree_attn_kernel<128>, &cfg) == cudaSuccess && n > 0)
      g_max_split = 16;
    cudaGetLastError();   // a refused query leaves the portable size
  });
  if (err != cudaSuccess) return fail(SUB_ECUDA, std::string("attn_init: ") + cudaGetErrorString(err));
  return SUB_OK;
}

int32_t launch_tree_attn(const AttnArgs& a, int n_split, cudaStream_t st) {
  SUB_CHECK_ARG(a.head_dim == 64 || a.head_dim == 128, "attn: head_dim must be 64 or 128");
  SUB_CHECK_ARG(a.n_heads_kv >= 1 && a.n_heads_q % a.n_heads_kv == 0, "attn: Hq % Hkv != 0");
  SUB_CHECK_ARG(a.page_size % 16 == 0 && a.page_size > 0, "attn: page_size % 16 != 0");
  SUB_CHECK_ARG(a.n_slots >= 0 && a.n_slots <= 16384, "attn: n_slots out of range");
  SUB_TRY(attn_init());
  SUB_CHECK_ARG((n_split >= 1 && n_split <= g_max_split) ||
                    (g_max_split == ATTN_MAX_SPLIT && n_split % ATTN_XCLUSTER == 0 &&
                     a.xpart && a.xm && a.xl && a.xcnt),
                "attn: bad split count");
  if (a.n_q == 0) return SUB_OK;
  const int G = a.n_heads_q / a.n_heads_kv;
  const int smem = attn_smem_bytes(a);
  SUB_CHECK_ARG(smem <= ATTN_MAX_SMEM, "attn: tree too large for the shared-memory bitmap");
  SUB_TRY(attn_init());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.n_q * G + ROWS - 1) / ROWS, a.n_heads_kv, n_split);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (n_split > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = n_split > ATTN_MAX_SPLIT ? ATTN_XCLUSTER : n_split;
    ++na;
  }
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (a.head_dim == 128) SUB_CUDA_TRY(cudaLaunchKernelEx(&cfg, tree_attn_kernel<128>, a));
  else SUB_CUDA_TRY(cudaLaunchKernelEx(&cfg, tree_attn_kernel<64>, a));
  return SUB_OK;
}

}  // namespace sub
