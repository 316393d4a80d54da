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
// shared memory, so no global scratch and no second launch are needed.
#include <mutex>
#include <cooperative_groups.h>
#include "attn.cuh"

namespace sub {

namespace {
constexpr int ROWS = 64, KT = 64, THREADS = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(pred ? 16 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
}  // namespace

// D = head_dim (64 or 128).  smem: Q [64][D], K/V double-buffered [2][64][D], bitmap.
template <int D>
__global__ void __launch_bounds__(THREADS) tree_attn_kernel(AttnArgs a) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + ROWS * D * 2;
  uint8_t* sV = sK + 2 * KT * D * 2;
  uint32_t* sBits = reinterpret_cast<uint32_t*>(sV + 2 * KT * D * 2);
  auto sw = [](int row, int ch) { return row * CH + (ch ^ (row & 7)); };

  // Programmatic dependent launch (early_reads): only Q and the K/V of the
  // query rows' own slots come from the kernel just before this one (the
  // q/k/v projection).  The tree (ancestors, depths), the page table, the
  // counters and every other key were written by kernels that finished before
  // that one's own predecessor did, so they are read before the wait.  This
  // holds because every kernel of the decode path signals its dependents only
  // from threads that have passed their own wait.  A caller of the public
  // entry point may have run anything just before, so there every read waits.
  if (!a.early_reads) pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kvh = blockIdx.y;
  const int G = a.n_heads_q / a.n_heads_kv;
  const int n_rows = a.n_q * G;
  const int row0 = blockIdx.x * ROWS;
  const int n_prefix = a.n_prefix_dev ? *a.n_prefix_dev : (int)a.n_prefix;
  const int64_t tree_base = a.tree_base_dev ? (int64_t)*a.tree_base_dev : a.tree_base;
  const int n_keys = n_prefix + a.n_slots;
  // this split's key range, whole tiles
  const int tiles_total = (n_keys + KT - 1) / KT;
  const int tiles_per = (tiles_total + gridDim.z - 1) / gridDim.z;
  const int t_begin = blockIdx.z * tiles_per;
  const int t_end = min(tiles_total, t_begin + tiles_per);

  const int q_lo = row0 / G;
  const int q_hi = min(a.n_q - 1, (row0 + ROWS - 1) / G);
  const int words = (a.n_slots + 31) / 32;

  // ---- visibility bitmaps of this CTA's queries ----
  // every ancestor entry and its query's depth are loaded together into
  // registers (one round trip), and set into the cleared bitmaps after the
  // barrier below
  constexpr int ANC_PER = 6;   // entries per thread per round
  const int nq = q_hi - q_lo + 1;
  const int n_anc = a.anc ? nq * a.anc_stride : 0;
  int anc_s[ANC_PER], anc_d[ANC_PER];
  if (a.anc) {
    for (int i = tid; i < nq * words; i += THREADS) sBits[i] = 0;
#pragma unroll
    for (int u = 0; u < ANC_PER; ++u) {
      const int i = tid + u * THREADS;
      anc_s[u] = -1;
      anc_d[u] = -1;
      if (i < n_anc) {
        const int qq = i / a.anc_stride;
        anc_s[u] = a.anc[(int64_t)(q_lo + qq) * a.anc_stride + i % a.anc_stride];
        anc_d[u] = a.depth[q_lo + qq];
      }
    }
  }
  const size_t head_stride = (size_t)a.page_size * D;
  const size_t page_stride = (size_t)a.n_heads_kv * head_stride;
  const size_t layer_off = (size_t)a.layer * a.n_pages * page_stride;
  auto key_pos = [&](int j) -> int64_t {
    return j < n_prefix ? (int64_t)j : tree_base + (j - n_prefix);
  };
  // element offset of every key row of a tile, resolved once per tile by KT
  // threads in parallel (page-table lookups), one tile ahead of its copy
  __shared__ int64_t sOff[2][KT];
  auto row_offsets = [&](int slot, int t) {
    if (tid < KT) {
      const int j = t * KT + tid;
      int64_t off = -1;
      if (t < t_end && j < n_keys) {
        const int64_t p = key_pos(j);
        const int page = a.page_table[p / a.page_size];
        off = (int64_t)(layer_off + (size_t)page * page_stride + (size_t)kvh * head_stride +
                        (size_t)(p % a.page_size) * D);
      }
      sOff[slot][tid] = off;
    }
  };
  auto load_kv = [&](int buf, int t) {
    (void)t;
    for (int c = tid; c < KT * CH; c += THREADS) {
      const int r = c / CH, ch = c % CH;
      const int64_t off = sOff[buf][r];
      const bool ok = off >= 0;
      const size_t src = ok ? (size_t)off + ch * 8 : 0;
      cp_async16(smem_u32(sK + buf * KT * D * 2 + sw(r, ch) * 16), a.k + src, ok);
      cp_async16(smem_u32(sV + buf * KT * D * 2 + sw(r, ch) * 16), a.v + src, ok);
    }
  };

  row_offsets(0, t_begin);
  row_offsets(1, t_begin + 1);
  __syncthreads();   // cleared bitmaps and the first row offsets are visible
  if (a.anc) {
    // entry j of query q counts for depths 0..depth[q]
    auto set_bit = [&](int i, int sv, int dv) {
      const int qq = i / a.anc_stride, j = i % a.anc_stride;
      if (j <= dv && sv >= 0 && sv < a.n_slots)
        atomicOr(&sBits[qq * words + (sv >> 5)], 1u << (sv & 31));
    };
#pragma unroll
    for (int u = 0; u < ANC_PER; ++u)
      if (tid + u * THREADS < n_anc) set_bit(tid + u * THREADS, anc_s[u], anc_d[u]);
    for (int i = tid + ANC_PER * THREADS; i < n_anc; i += THREADS) {   // wider trees
      const int qq = i / a.anc_stride;
      set_bit(i, a.anc[(int64_t)(q_lo + qq) * a.anc_stride + i % a.anc_stride],
              a.depth[q_lo + qq]);
    }
  }
  // the first tile before the wait unless it holds a slot of the query rows
  // (keys n_prefix + chain_slot0 .. + n_q - 1 are this pass's own K/V)
  const int fresh_lo = (n_prefix + a.chain_slot0) / KT;
  const int fresh_hi = (n_prefix + a.chain_slot0 + a.n_q - 1) / KT;
  const bool first_fresh = t_begin >= fresh_lo && t_begin <= fresh_hi;
  if (t_begin < t_end && !first_fresh) load_kv(0, t_begin);
  pdl_wait();
  if (t_begin < t_end && first_fresh) load_kv(0, t_begin);
  cp_commit();   // group: the first K/V tile
  // ---- Q tile ----
  const size_t q_row_stride = (size_t)a.n_heads_q * D;
  for (int c = tid; c < ROWS * CH; c += THREADS) {
    const int r = c / CH, ch = c % CH;
    const int gr = row0 + r;
    const bool ok = gr < n_rows;
    const int q = ok ? gr / G : 0, h = ok ? gr % G : 0;
    const uint16_t* src = a.Q + (size_t)q * q_row_stride + (size_t)(kvh * G + h) * D + ch * 8;
    cp_async16(smem_u32(sQ + sw(r, ch) * 16), src, ok);
  }
  cp_commit();   // group: Q

  // per-lane rows: g and g+8 of this warp's 16
  const int g = lane >> 2, tig = lane & 3;
  const int wrow = warp * 16;
  int rq[2];      // query index of each of the lane's two rows (-1 if none)
  int rslot[2];   // chain mode: the query's own slot
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gr = row0 + wrow + g + 8 * h;
    rq[h] = gr < n_rows ? gr / G : -1;
    rslot[h] = rq[h] >= 0 ? a.chain_slot0 + rq[h] : -1;
  }

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  cp_wait<0>();   // Q and the first K/V tile landed
  __syncthreads();
  uint32_t qf[D / 16][4];
  {
    const uint32_t qb = smem_u32(sQ);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ldsm_x4(qb + sw(wrow + (lane & 15), kk * 2 + (lane >> 4)) * 16, qf[kk][0], qf[kk][1],
              qf[kk][2], qf[kk][3]);
  }
  const float sl2 = a.scale * 1.4426950408889634f;   // scores in log2 units

  for (int t = t_begin; t < t_end; ++t) {
    const int buf = (t - t_begin) & 1;
    if (t + 1 < t_end) load_kv(buf ^ 1, t + 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();

    const uint32_t kb = smem_u32(sK + buf * KT * D * 2);
    const uint32_t vb = smem_u32(sV + buf * KT * D * 2);
    float s[KT / 8][4];
#pragma unroll
    for (int j = 0; j < KT / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int jj = 0; jj < KT / 16; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + sw(jj * 16 + (lane & 7) + ((lane >> 4) << 3), kk * 2 + ((lane >> 3) & 1)) * 16,
                b0, b1, b2, b3);
        mma_bf16_16816(s[2 * jj], qf[kk], b0, b1);
        mma_bf16_16816(s[2 * jj + 1], qf[kk], b2, b3);
      }
    // visibility of the tile's 64 keys for the lane's two rows, as two 32-bit
    // masks per row: a key of the prefix is seen by every query, a tree slot
    // by the queries it is an ancestor of (chain: the slots up to the query's
    // own), keys past n_keys by none.  Rows past the queries (padding) see the
    // whole tile; their results are never written.
    const int key0 = t * KT;
    uint32_t vm[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t lo = ~0u, hi = ~0u;
      if (key0 + KT > n_prefix && rq[h] >= 0) {
        const int sl0 = key0 - n_prefix;   // slot of the tile's first key (> -KT)
        if (a.anc) {
          const uint32_t* bits = sBits + (rq[h] - q_lo) * words;
          auto word = [&](int wi) -> uint32_t {   // prefix keys sit at negative slots
            return wi < 0 ? ~0u : (wi < words ? bits[wi] : 0u);
          };
          const int w0 = sl0 >> 5, off = sl0 & 31;   // floor division
          const uint32_t a0 = word(w0), a1 = word(w0 + 1), a2 = word(w0 + 2);
          lo = __funnelshift_r(a0, a1, off);
          hi = __funnelshift_r(a1, a2, off);
        } else {
          const int cnt = rslot[h] - sl0 + 1;   // keys key0 .. key0 + cnt - 1 are seen
          lo = cnt >= 32 ? ~0u : (cnt <= 0 ? 0u : (1u << cnt) - 1u);
          hi = cnt >= 64 ? ~0u : (cnt <= 32 ? 0u : (1u << (cnt - 32)) - 1u);
        }
        const int nv = n_keys - key0;   // >= 1 keys of the tile exist
        if (nv < 64) {
          lo &= nv >= 32 ? ~0u : (1u << nv) - 1u;
          hi &= nv <= 32 ? 0u : (1u << (nv - 32)) - 1u;
        }
      }
      vm[h][0] = lo;
      vm[h][1] = hi;
    }
    // mask, scale, online softmax
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < KT / 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        const int kk = (j & 3) * 8 + 2 * tig + (e & 1);   // bit within the 32-key half j / 4
        const bool vis = (vm[h][j >> 2] >> kk) & 1u;
        const float v = vis ? s[j][e] * sl2 : -INFINITY;
        s[j][e] = v;
        tmax[h] = fmaxf(tmax[h], v);
      }
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
      tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
      const float m_new = fmaxf(m_run[h], tmax[h]);
      corr[h] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[h] - m_new);
      m_run[h] = m_new;
    }
    float tsum[2] = {0.f, 0.f};
    // P as the A operand in two bf16 parts, hi = bf16(p) and lo = bf16(p - hi)
    // (p - hi is exact in fp32), so that P.V keeps p to ~2^-17 relative: one
    // bf16 rounding of P (2^-9) shifts a layer's output by ~0.5% against the
    // exact softmax, which the decode's token choices cannot absorb
    uint32_t pa[KT / 16][4], pl[KT / 16][4];
#pragma unroll
    for (int j = 0; j < KT / 8; ++j) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        p[e] = (m_run[h] == -INFINITY) ? 0.f : exp2f(s[j][e] - m_run[h]);
        tsum[h] += p[e];
      }
      // n8 tiles 2i, 2i+1 form k16 step i
      const int r0 = (j & 1) ? 2 : 0;
      const uint32_t h01 = pack_bf16x2(p[0], p[1]), h23 = pack_bf16x2(p[2], p[3]);
      pa[j >> 1][r0] = h01;
      pa[j >> 1][r0 + 1] = h23;
      pl[j >> 1][r0] = pack_bf16x2(p[0] - bf16lo(h01), p[1] - bf16hi(h01));
      pl[j >> 1][r0 + 1] = pack_bf16x2(p[2] - bf16lo(h23), p[3] - bf16hi(h23));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      tsum[h] += __shfl_xor_sync(0xffffffffu, tsum[h], 1);
      tsum[h] += __shfl_xor_sync(0xffffffffu, tsum[h], 2);
      l_run[h] = l_run[h] * corr[h] + tsum[h];
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= corr[0]; o[i][1] *= corr[0];
      o[i][2] *= corr[1]; o[i][3] *= corr[1];
    }
#pragma unroll
    for (int kk = 0; kk < KT / 16; ++kk)
#pragma unroll
      for (int dd = 0; dd < D / 16; ++dd) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + sw(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), dd * 2 + (lane >> 4)) * 16,
                  b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dd], pa[kk], b0, b1);
        mma_bf16_16816(o[2 * dd + 1], pa[kk], b2, b3);
        mma_bf16_16816(o[2 * dd], pl[kk], b0, b1);
        mma_bf16_16816(o[2 * dd + 1], pl[kk], b2, b3);
      }
    row_offsets(buf, t + 2);
    __syncthreads();   // buffer reuse by the next prefetch; row offsets of tile t + 2
  }

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
  const int S = (int)gridDim.z;
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
  if (act) sWl[mi * S + ms2] = w_peer * (den > 0.f ? 1.f / den : 0.f);
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
    const int q = gr / G, hh = gr % G;
    const size_t orow = (size_t)q * a.n_heads_q + kvh * G + hh;
    *reinterpret_cast<uint2*>(a.O + orow * D + c) = make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
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

int attn_pick_splits(const AttnArgs& a, int n_keys_hint) {
  if (attn_init() != SUB_OK) return 1;
  const int G = a.n_heads_q / a.n_heads_kv;
  const int blocks = (a.n_q * G + ROWS - 1) / ROWS * a.n_heads_kv;
  const int tiles = (n_keys_hint + KT - 1) / KT;
  int s = (2 * 152 + blocks - 1) / blocks;
  s = std::max(1, std::min(s, std::min(tiles, g_max_split)));
  return s;
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
  SUB_CHECK_ARG(n_split >= 1 && n_split <= g_max_split, "attn: bad split count");
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
    attr[na].val.clusterDim.z = n_split;
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
