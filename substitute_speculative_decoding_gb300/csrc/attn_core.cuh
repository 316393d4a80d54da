// The main loop of tree-masked attention over the paged KV cache (see attn.cu
// for the method): one CTA's 64 rows of one KV head over a split of the key
// tiles, on mma.sync with an online softmax, as a device function whose
// caller chooses the barrier among the 128 participating threads and what to
// do with the partial results (attn.cu merges them inside a cluster).
#pragma once
#include "attn.cuh"

namespace sub {

namespace attn_detail {
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

// The main loop of one CTA: the 64 rows from row0 on ((query, head-in-group)
// pairs of KV head kvh) over this split's share of the key tiles; threads
// 0..127 take part (sync() is a barrier among them) and each leaves its two
// rows' running max, sum and unnormalised output in m_run, l_run and o.
// D = head_dim (64 or 128).  smem: Q [64][D], K/V double-buffered [2][64][D], bitmap.
template <int D, class Sync>
__device__ __forceinline__ void attn_main(const AttnArgs& a, int kvh, int row0, int split,
                                          int n_split, uint8_t* smem, Sync sync,
                                          float (&o)[D / 8][4], float (&m_run)[2],
                                          float (&l_run)[2]) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
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
  const int G = a.n_heads_q / a.n_heads_kv;
  const int n_rows = a.n_q * G;
  const int n_prefix = a.n_prefix_dev ? *a.n_prefix_dev : (int)a.n_prefix;
  const int64_t tree_base = a.tree_base_dev ? (int64_t)*a.tree_base_dev : a.tree_base;
  const int n_keys = n_prefix + a.n_slots;
  // this split's key range, whole tiles
  const int tiles_total = (n_keys + KT - 1) / KT;
  const int tiles_per = (tiles_total + n_split - 1) / n_split;
  const int t_begin = split * tiles_per;
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
  sync();   // cleared bitmaps and the first row offsets are visible
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

  m_run[0] = m_run[1] = -INFINITY;
  l_run[0] = l_run[1] = 0.f;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  cp_wait<0>();   // Q and the first K/V tile landed
  sync();
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
    sync();

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
    sync();   // buffer reuse by the next prefetch; row offsets of tile t + 2
  }
}

}  // namespace attn_detail

using attn_detail::attn_main;
using attn_detail::KT;
using attn_detail::ROWS;
using attn_detail::THREADS;

}  // namespace sub
