// Warp-level GEMV kernels (bf16 and int4 weights), see gemv.cuh.
//
// A CTA owns RT row tiles (16 rows each, two per lane: g and g + 8) over one
// split of K.  Each warp keeps U steps of weights and activations in flight
// with a rolling register prefetch; the first U weight steps are requested
// before the programmatic-launch wait.  Splits of K over CTAs (grid.y) meet in
// a scratch buffer and the last split of a unit adds them in split order.
#include <algorithm>
#include "gemv.cuh"

namespace sub {

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

constexpr int WK = 4;   // warps per CTA, splitting the CTA's K range

// Activations are written by the previous kernel of the stream: L2-coherent
// loads that the compiler may not hoist above the programmatic-launch wait.
__device__ __forceinline__ uint4 ldcg_v4(const uint16_t* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}

// Rows of tile t of this CTA: (segment, local row of fragment row g, local
// row of fragment row g + 8); the fragment rows are lo + g and hi + g.
struct TileRows {
  int seg, lo, hi;
};

template <int EPI, int RT>
__device__ __forceinline__ TileRows tile_rows(const GemvArgs& a, int t) {
  TileRows r;
  if constexpr (EPI == EPI_GLU) {
    r.seg = t / RT;
    r.lo = (blockIdx.x * RT + t % RT) * 16;
    r.hi = r.lo + 8;
  } else if constexpr (EPI == EPI_QKV) {
    const int D = a.qkv.head_dim, per_head = D / 16;
    const int tq = a.qkv.n_heads_q * per_head, tk = a.qkv.n_heads_kv * per_head;
    const int vt = blockIdx.x;
    if (vt < tq + tk) {
      const int v = vt < tq ? vt : vt - tq;
      r.seg = vt < tq ? 0 : 1;
      r.lo = (v / per_head) * D + 8 * (v % per_head);
      r.hi = r.lo + D / 2;            // RoPE partner rows in the same fragment
    } else {
      r.seg = 2;
      r.lo = (vt - tq - tk) * 16;
      r.hi = r.lo + 8;
    }
  } else {
    const int vrow = (blockIdx.x * RT + t) * 16;
    int seg = 0, start = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i)
      if (seg < a.n_seg - 1 && vrow >= a.seg_end[seg]) { start = a.seg_end[seg]; ++seg; }
    r.seg = seg;
    r.lo = vrow - start;
    r.hi = r.lo + 8;
  }
  return r;
}

template <int EPI>
__device__ __forceinline__ int seg_rows(const GemvArgs& a, int seg) {
  if constexpr (EPI == EPI_GLU) return a.N;
  return a.seg_end[seg] - (seg ? a.seg_end[seg - 1] : 0);
}

// K columns of each split: bf16 steps of 32, int4 groups of 64, whole U batches.
template <bool W4, int U>
__host__ __device__ inline int split_units(int K, int ks) {
  const int total = W4 ? (K + 63) / 64 : (K + 31) / 32;
  return ((total + ks - 1) / ks + U - 1) / U * U;
}

// One lane's 16 codes of group gi (elements 16 * tig .. 16 * tig + 15 of the
// group) as two int4-layout words; row points at the row's first group.
template <int QB>
__device__ __forceinline__ uint2 load_codes(const char* row, int gi, int tig) {
  const char* grp = row + (int64_t)gi * (8 * QB);
  if constexpr (QB == 4) {
    return ldg_nc_v2(grp + tig * 8);
  } else {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(grp + tig * 4));
    uint2 r = make_uint2(spread2(w), spread2(w >> 16));
    if constexpr (QB == 3) {
      const uint32_t h = __ldg(reinterpret_cast<const uint16_t*>(grp + 16 + tig * 2));
      r.x |= spread1(h) << 2;
      r.y |= spread1(h >> 8) << 2;
    }
    return r;
  }
}

template <bool W4, int MT, int RT, int EPI, int U, int QB = 4>
__global__ void __launch_bounds__(WK * 32)
gemv_kernel(GemvArgs a) {
  constexpr bool GLU = (EPI == EPI_GLU);
  constexpr int NT = GLU ? 2 * RT : RT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int K = a.K;
  const int G = (K + 63) / 64;
  const int ks = gridDim.y;

  // this CTA's K range, in steps of 32 (bf16) or groups of 64 (int4)
  const int total_u = W4 ? G : (K + 31) / 32;
  const int per_split = split_units<W4, U>(K, ks);
  const int r_begin = blockIdx.y * per_split, r_end = min(total_u, r_begin + per_split);
  const int per = ((r_end - r_begin + WK - 1) / WK + U - 1) / U * U;
  const int u_begin = r_begin + warp * per, u_end = min(r_end, u_begin + per);

  // ---- per-tile row pointers (two rows per lane: g and g + 8) ----
  const char* rp0[NT];
  const char* rp1[NT];
  const uint16_t* sp0[NT];
  const uint16_t* sp1[NT];
  const uint16_t* zp0[NT];
  const uint16_t* zp1[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const TileRows tr = tile_rows<EPI, RT>(a, t);
    const int nrows = seg_rows<EPI>(a, tr.seg);
    const int r0 = min(tr.lo + g, nrows - 1);
    const int r1 = min(tr.hi + g, nrows - 1);
    const char* base = reinterpret_cast<const char*>(a.W[tr.seg]);
    if constexpr (W4) {
      rp0[t] = base + (int64_t)r0 * G * (8 * QB);
      rp1[t] = base + (int64_t)r1 * G * (8 * QB);
      sp0[t] = a.S[tr.seg] + (int64_t)r0 * G;
      sp1[t] = a.S[tr.seg] + (int64_t)r1 * G;
      zp0[t] = a.Z[tr.seg] + (int64_t)r0 * G;
      zp1[t] = a.Z[tr.seg] + (int64_t)r1 * G;
    } else {
      rp0[t] = base + ((int64_t)r0 * K + tig * 8) * 2;
      rp1[t] = base + ((int64_t)r1 * K + tig * 8) * 2;
    }
  }
  const uint16_t* xp[MT];
  bool xok[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = mt * 8 + g;
    xok[mt] = m < a.M;
    xp[mt] = a.X + (int64_t)(xok[mt] ? m : 0) * a.ldx;
  }

  float acc[NT][MT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[t][mt][j] = 0.f;

  if constexpr (!W4) {
    // ------------------------------------------------ bf16 weights ----
    uint4 w0[U][NT], w1[U][NT], xv[U][MT];
    auto load_w = [&](int u, int s) {
      const bool ok = s < u_end && s * 32 + tig * 8 < K;   // K % 8 == 0: whole chunks
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        w0[u][t] = ok ? ldg_nc_v4(rp0[t] + (int64_t)s * 64) : make_uint4(0, 0, 0, 0);
        w1[u][t] = ok ? ldg_nc_v4(rp1[t] + (int64_t)s * 64) : make_uint4(0, 0, 0, 0);
      }
    };
    auto load_x = [&](int u, int s) {
      const int k = s * 32 + tig * 8;
      const bool ok = s < u_end && k < K;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        xv[u][mt] = (ok && xok[mt]) ? ldcg_v4(xp[mt] + k) : make_uint4(0, 0, 0, 0);
    };
#pragma unroll
    for (int u = 0; u < U; ++u) load_w(u, u_begin + u);   // weights before the wait
    pdl_wait();
#pragma unroll
    for (int u = 0; u < U; ++u) load_x(u, u_begin + u);
    for (int s = u_begin; s < u_end; s += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t A0[4] = {w0[u][t].x, w1[u][t].x, w0[u][t].y, w1[u][t].y};
            const uint32_t A1[4] = {w0[u][t].z, w1[u][t].z, w0[u][t].w, w1[u][t].w};
            mma_bf16_16816(acc[t][mt], A0, xv[u][mt].x, xv[u][mt].y);
            mma_bf16_16816(acc[t][mt], A1, xv[u][mt].z, xv[u][mt].w);
          }
        load_w(u, s + U + u);
        load_x(u, s + U + u);
      }
    }
  } else {
    // ------------------------------------------------ int4 weights ----
    // scales/zeros of 4 consecutive groups in one 8-byte load when rows allow
    const bool sz_vec = (G % 4 == 0);
    const uint32_t ONES = 0x3f803f80u;
    const uint32_t ONES_A[4] = {ONES, ONES, ONES, ONES};
    static_assert(U % 4 == 0, "int4 batches are whole 4-group scale loads");
    constexpr int UB = U / 4;
    uint2 q0[U][NT], q1[U][NT];
    uint2 sv0[UB][NT], sv1[UB][NT], zv0[UB][NT], zv1[UB][NT];
    uint16_t ss0[U][NT], ss1[U][NT], zs0[U][NT], zs1[U][NT];
    uint4 xa[U][MT], xb[U][MT];
    auto load_q = [&](int u, int gi) {
      const bool ok = gi < u_end;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        q0[u][t] = ok ? load_codes<QB>(rp0[t], gi, tig) : make_uint2(0, 0);
        q1[u][t] = ok ? load_codes<QB>(rp1[t], gi, tig) : make_uint2(0, 0);
        if (!sz_vec) {
          ss0[u][t] = ok ? __ldg(sp0[t] + gi) : 0;
          ss1[u][t] = ok ? __ldg(sp1[t] + gi) : 0;
          zs0[u][t] = ok ? __ldg(zp0[t] + gi) : 0;
          zs1[u][t] = ok ? __ldg(zp1[t] + gi) : 0;
        }
      }
      // groups gi - 3 .. gi in one 8-byte load (gi - 3 is a multiple of 4), issued
      // with the last of the four slots that use them, so the rolling reload
      // never overwrites scales of the batch in progress
      if (sz_vec && (u & 3) == 3) {
        const int b = u >> 2, g4 = gi - 3;
        const bool ok4 = g4 < u_end;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          sv0[b][t] = ok4 ? __ldg(reinterpret_cast<const uint2*>(sp0[t] + g4)) : make_uint2(0, 0);
          sv1[b][t] = ok4 ? __ldg(reinterpret_cast<const uint2*>(sp1[t] + g4)) : make_uint2(0, 0);
          zv0[b][t] = ok4 ? __ldg(reinterpret_cast<const uint2*>(zp0[t] + g4)) : make_uint2(0, 0);
          zv1[b][t] = ok4 ? __ldg(reinterpret_cast<const uint2*>(zp1[t] + g4)) : make_uint2(0, 0);
        }
      }
    };
    auto load_x = [&](int u, int gi) {
      const bool ok = gi < u_end;
      const int k = gi * 64 + tig * 16;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        xa[u][mt] = (ok && xok[mt] && k < K) ? ldcg_v4(xp[mt] + k) : make_uint4(0, 0, 0, 0);
        xb[u][mt] = (ok && xok[mt] && k + 8 < K) ? ldcg_v4(xp[mt] + k + 8) : make_uint4(0, 0, 0, 0);
      }
    };
#pragma unroll
    for (int u = 0; u < U; ++u) load_q(u, u_begin + u);   // weights before the wait
    pdl_wait();
#pragma unroll
    for (int u = 0; u < U; ++u) load_x(u, u_begin + u);
    for (int gi0 = u_begin; gi0 < u_end; gi0 += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        // B fragments: pairs (k, k+4) to match the nibble pairs of one packed word
        uint32_t b[MT][4][2];
        float sx[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          b[mt][0][0] = __byte_perm(xa[u][mt].x, xa[u][mt].z, 0x5410);
          b[mt][0][1] = __byte_perm(xa[u][mt].x, xa[u][mt].z, 0x7632);
          b[mt][1][0] = __byte_perm(xa[u][mt].y, xa[u][mt].w, 0x5410);
          b[mt][1][1] = __byte_perm(xa[u][mt].y, xa[u][mt].w, 0x7632);
          b[mt][2][0] = __byte_perm(xb[u][mt].x, xb[u][mt].z, 0x5410);
          b[mt][2][1] = __byte_perm(xb[u][mt].x, xb[u][mt].z, 0x7632);
          b[mt][3][0] = __byte_perm(xb[u][mt].y, xb[u][mt].w, 0x5410);
          b[mt][3][1] = __byte_perm(xb[u][mt].y, xb[u][mt].w, 0x7632);
#pragma unroll
          for (int j = 0; j < 4; ++j) sx[mt][j] = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) mma_bf16_16816(sx[mt], ONES_A, b[mt][i][0], b[mt][i][1]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          // scale and 128 + zero of rows g and g + 8 for group gi0 + u
          uint32_t a0s, a1s, b0z, b1z;
          if (sz_vec) {
            const int bb = u >> 2;
            const uint32_t ws0 = (u & 2) ? sv0[bb][t].y : sv0[bb][t].x;
            const uint32_t ws1 = (u & 2) ? sv1[bb][t].y : sv1[bb][t].x;
            const uint32_t wz0 = (u & 2) ? zv0[bb][t].y : zv0[bb][t].x;
            const uint32_t wz1 = (u & 2) ? zv1[bb][t].y : zv1[bb][t].x;
            a0s = (u & 1) ? (ws0 >> 16) : (ws0 & 0xffffu);
            a1s = (u & 1) ? (ws1 >> 16) : (ws1 & 0xffffu);
            b0z = (u & 1) ? (wz0 >> 16) : (wz0 & 0xffffu);
            b1z = (u & 1) ? (wz1 >> 16) : (wz1 & 0xffffu);
          } else {
            a0s = ss0[u][t]; a1s = ss1[u][t]; b0z = zs0[u][t]; b1z = zs1[u][t];
          }
          const float sr0 = __uint_as_float(a0s << 16), sr1 = __uint_as_float(a1s << 16);
          const float zr0 = 128.0f + __uint_as_float(b0z << 16);
          const float zr1 = 128.0f + __uint_as_float(b1z << 16);
          // nibble pairs (n_i, n_{i+4}) of each word -> bf16x2 (128 + q); mma i
          // reads word i/2 of each row: pairs (0,4),(1,5) for even i and
          // (2,6),(3,7) for odd i; the B fragments pair K the same way
          uint32_t A[4][4];
          {
            const uint32_t a0 = q0[u][t].x, a1 = q0[u][t].y;   // row g: words 0, 1
            const uint32_t c0 = q1[u][t].x, c1 = q1[u][t].y;   // row g + 8
            const uint32_t NIB = 0x000f000fu, E = 0x43004300u;
            A[0][0] = (a0 & NIB) | E;         A[0][2] = ((a0 >> 4) & NIB) | E;
            A[0][1] = (c0 & NIB) | E;         A[0][3] = ((c0 >> 4) & NIB) | E;
            A[1][0] = ((a0 >> 8) & NIB) | E;  A[1][2] = ((a0 >> 12) & NIB) | E;
            A[1][1] = ((c0 >> 8) & NIB) | E;  A[1][3] = ((c0 >> 12) & NIB) | E;
            A[2][0] = (a1 & NIB) | E;         A[2][2] = ((a1 >> 4) & NIB) | E;
            A[2][1] = (c1 & NIB) | E;         A[2][3] = ((c1 >> 4) & NIB) | E;
            A[3][0] = ((a1 >> 8) & NIB) | E;  A[3][2] = ((a1 >> 12) & NIB) | E;
            A[3][1] = ((c1 >> 8) & NIB) | E;  A[3][3] = ((c1 >> 12) & NIB) | E;
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t Ai[4] = {A[i][0], A[i][1], A[i][2], A[i][3]};
              mma_bf16_16816(p, Ai, b[mt][i][0], b[mt][i][1]);
            }
            // rows g (p0, p1) and g+8 (p2, p3); tokens 2tig (p0, p2), 2tig+1 (p1, p3)
            acc[t][mt][0] = fmaf(sr0, fmaf(-zr0, sx[mt][0], p[0]), acc[t][mt][0]);
            acc[t][mt][1] = fmaf(sr0, fmaf(-zr0, sx[mt][1], p[1]), acc[t][mt][1]);
            acc[t][mt][2] = fmaf(sr1, fmaf(-zr1, sx[mt][2], p[2]), acc[t][mt][2]);
            acc[t][mt][3] = fmaf(sr1, fmaf(-zr1, sx[mt][3], p[3]), acc[t][mt][3]);
          }
        }
        load_q(u, gi0 + U + u);
        load_x(u, gi0 + U + u);
      }
    }
  }

  // the next kernel may launch now and stream its weights during this epilogue
  pdl_trigger();
  // ---- cross-warp reduction in a fixed order, then the epilogue ----
  constexpr int PER_WARP = NT * MT * 4 * 32;
  __shared__ float red[WK * PER_WARP];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        red[warp * PER_WARP + ((t * MT + mt) * 4 + j) * 32 + lane] = acc[t][mt][j];
  __syncthreads();
  __shared__ float tot_s[PER_WARP];
  for (int e = threadIdx.x; e < PER_WARP; e += WK * 32) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < WK; ++w) v += red[w * PER_WARP + e];
    tot_s[e] = v;
  }
  if (ks > 1) {
    // split of K over CTAs: park this split's sums, the last split of the unit adds all
    __shared__ unsigned int s_split_last;
    __syncthreads();
    float* mine = a.split_part + ((size_t)blockIdx.x * ks + blockIdx.y) * PER_WARP;
    for (int e = threadIdx.x; e < PER_WARP; e += WK * 32) mine[e] = tot_s[e];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      s_split_last = (atomicAdd(a.split_cnt + blockIdx.x, 1u) == (unsigned)ks - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_split_last) return;
    __threadfence();
    const float* all = a.split_part + (size_t)blockIdx.x * ks * PER_WARP;
    for (int e = threadIdx.x; e < PER_WARP; e += WK * 32) {
      float v = 0.f;
      for (int y = 0; y < ks; ++y) v += __ldcg(all + (size_t)y * PER_WARP + e);
      tot_s[e] = v;
    }
    if (threadIdx.x == 0) a.split_cnt[blockIdx.x] = 0u;
  }
  // factored RMSNorm of the input: scale each token's sums by its row scale
  __shared__ float s_r[16];
  if (a.xscale.partial)
    for (int m = warp; m < a.M; m += WK) {
      const float r = row_scale(a.xscale, m, lane);
      if (lane == 0) s_r[m] = r;
    }
  __syncthreads();
  auto total = [&](int e, int tok) {
    const float v = tot_s[e];
    return a.xscale.partial ? v * s_r[tok] : v;
  };

  if constexpr (EPI == EPI_QKV) {
    // element e = (mt * 4 + j) * 32 + ln; j in {0,1}: rows g (lo), e + 64: rows g + 8 (hi)
    const QkvOut& qo = a.qkv;
    const TileRows tr = tile_rows<EPI, RT>(a, 0);
    const int D = qo.head_dim, half = D / 2;
    const int64_t base = qo.base_dev ? (int64_t)*qo.base_dev : qo.base;
    const size_t head_stride = (size_t)qo.page_size * D;
    const size_t page_stride = (size_t)qo.n_heads_kv * head_stride;
    const size_t layer_off = (size_t)qo.layer * qo.n_pages * page_stride;
    for (int h = threadIdx.x; h < MT * 2 * 32; h += WK * 32) {
      const int ln = h & 31, j = (h >> 5) & 1, mt = h >> 6;
      const int e = (mt * 4 + j) * 32 + ln;
      const int gg = ln >> 2, tg = ln & 3;
      const int tok = mt * 8 + 2 * tg + j;
      if (tok >= a.M) continue;
      const float vlo = total(e, tok), vhi = total(e + 64, tok);
      const int64_t kvpos = base + qo.slot0 + tok;
      const size_t slot_off = layer_off + (size_t)qo.page_table[kvpos / qo.page_size] * page_stride +
                              (size_t)(kvpos % qo.page_size) * D;
      if (tr.seg < 2) {
        const int head = tr.lo / D;
        const int i = tr.lo % D + gg;   // index within the first half
        const int64_t pos = base + (qo.depth ? qo.depth[tok] : qo.slot0 + tok);
        const float2 cs = qo.rope[(pos < qo.max_pos ? pos : qo.max_pos - 1) * half + i];
        const float y1 = vlo * cs.x - vhi * cs.y;
        const float y2 = vhi * cs.x + vlo * cs.y;
        uint16_t* dst = tr.seg == 0
                            ? qo.q_out + ((size_t)tok * qo.n_heads_q + head) * D
                            : qo.k_cache + slot_off + (size_t)head * head_stride;
        dst[i] = f32_to_bf16_bits(y1);
        dst[i + half] = f32_to_bf16_bits(y2);
      } else {
        const int rlo = tr.lo + gg, rhi = tr.hi + gg;
        qo.v_cache[slot_off + (size_t)(rlo / D) * head_stride + rlo % D] = f32_to_bf16_bits(vlo);
        qo.v_cache[slot_off + (size_t)(rhi / D) * head_stride + rhi % D] = f32_to_bf16_bits(vhi);
      }
    }
    return;
  }

  constexpr int OUT_ELEMS = RT * MT * 4 * 32;
  for (int e = threadIdx.x; e < OUT_ELEMS; e += WK * 32) {
    // e = ((t * MT + mt) * 4 + j) * 32 + ln, t < RT
    const int ln = e & 31;
    const int j = (e >> 5) & 3;
    const int mt = (e >> 7) % MT;
    const int t = (e >> 7) / MT;
    const int gg = ln >> 2, tg = ln & 3;
    const int row = (blockIdx.x * RT + t) * 16 + gg + ((j & 2) ? 8 : 0);
    const int tok = mt * 8 + 2 * tg + (j & 1);
    if (row >= a.N || tok >= a.M) continue;
    const float v = total(e, tok);
    const int64_t o = (int64_t)tok * a.ldy + row;
    if constexpr (EPI == EPI_BF16) {
      reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(v);
    } else if constexpr (EPI == EPI_F32) {
      reinterpret_cast<float*>(a.Y)[o] = v;
    } else if constexpr (EPI == EPI_RESID) {
      float* yp = reinterpret_cast<float*>(a.Y) + o;
      const float xn = *yp + v;
      *yp = xn;
      if (a.norm.xn)   // next RMSNorm input, factored: bf16(x * gain)
        a.norm.xn[o] = f32_to_bf16_bits(xn * bf16_bits_to_f32(a.norm.gain[row]));
    } else {
      const float vu = total(e + RT * MT * 4 * 32, tok);   // same element of the 'up' tile
      reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(silu_f(v) * vu);
    }
  }

  if constexpr (EPI == EPI_RESID) {
    // next RMSNorm: per 16-row tile of this CTA, each token's sum of squares
    const NormOut& no = a.norm;
    if (!no.xn) return;
    const float* Y = reinterpret_cast<const float*>(a.Y);
    __syncthreads();   // this CTA's residual rows are written
    if (warp == 0 && lane < a.M) {
#pragma unroll
      for (int t = 0; t < RT; ++t) {
        const int row0 = (blockIdx.x * RT + t) * 16;
        if (row0 >= a.N) continue;
        float v[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
          v[r] = row0 + r < a.N ? __ldcg(Y + (int64_t)lane * a.ldy + row0 + r) : 0.f;
        float ss = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) ss = fmaf(v[r], v[r], ss);
        no.partial[(row0 / 16) * 16 + lane] = ss;
      }
    }
  }
}

// ------------------------------------------------------------------ launch --
static int pick_rt(const GemvArgs& a, int epi) {
  if (epi == EPI_GLU || epi == EPI_QKV) return 1;
  bool rt2 = a.N >= 32 * 152;
  for (int i = 0; i < a.n_seg; ++i) {
    const int start = i ? a.seg_end[i - 1] : 0;
    if ((a.seg_end[i] - start) % 32) rt2 = false;
  }
  return rt2 ? 2 : 1;
}

int gemv_grid(const GemvArgs& a, int epi) {
  if (epi == EPI_QKV) return a.N / 16;
  const int rt = pick_rt(a, epi);
  return (a.N + 16 * rt - 1) / (16 * rt);
}

// Splits of K over CTAs: each warp walks its K range in batches of U loads
// and pays about one memory latency per batch, so long K with few row units
// is latency-chained: aim at about 3 batches per warp when the row units
// alone leave fewer than 8 CTAs per SM.
static int pick_ksplit(const GemvArgs& a, bool w4, int units) {
  if (units >= 8 * 152) return 1;
  const int U = 4;
  const int batches = w4 ? ((a.K + 63) / 64 + U - 1) / U : ((a.K + 31) / 32 + U - 1) / U;
  int ks = (batches + 4 * 3 - 1) / (4 * 3);
  ks = std::max(1, std::min(ks, 8));
  while (ks > 1 && units * ks > 16 * 152) --ks;
  return ks;
}

int gemv_ksplit(const GemvArgs& a, bool is_w4, int epi) {
  return pick_ksplit(a, is_w4, gemv_grid(a, epi));
}

template <bool W4, int MT, int RT, int EPI, int QB>
static int32_t launch_cfg(const GemvArgs& a_in, cudaStream_t st) {
  constexpr int U = 4;
  constexpr int NT = (EPI == EPI_GLU) ? 2 * RT : RT;
  constexpr int PER = NT * MT * 4 * 32;
  GemvArgs a = a_in;
  const int units = gemv_grid(a, EPI);
  int ks = (a.split_part && a.split_cnt) ? pick_ksplit(a, W4, units) : 1;
  while (ks > 1 && ((size_t)units * ks * PER > a.split_cap || units > a.split_cnt_cap)) --ks;
  a.ksplit = ks;
  SUB_CUDA_TRY(launch_k(gemv_kernel<W4, MT, RT, EPI, U, QB>, dim3(units, ks), dim3(WK * 32), 0, st,
                        a));
  return SUB_OK;
}

// 2- and 3-bit codes (QB) run one row tile per warp only.
template <bool W4, int MT, int EPI, int QB>
static int32_t launch_rt(const GemvArgs& a, cudaStream_t st) {
  if constexpr (EPI == EPI_GLU || EPI == EPI_QKV || QB != 4) {
    return launch_cfg<W4, MT, 1, EPI, QB>(a, st);
  } else {
    if (pick_rt(a, EPI) == 2) return launch_cfg<W4, MT, 2, EPI, QB>(a, st);
    return launch_cfg<W4, MT, 1, EPI, QB>(a, st);
  }
}

template <bool W4, int EPI, int QB>
static int32_t launch_mt(const GemvArgs& a, cudaStream_t st) {
  if (a.M <= 8) return launch_rt<W4, 1, EPI, QB>(a, st);
  return launch_rt<W4, 2, EPI, QB>(a, st);
}

template <bool W4, int QB>
static int32_t launch_epi(const GemvArgs& a, int epi, cudaStream_t st) {
  switch (epi) {
    case EPI_BF16: return launch_mt<W4, EPI_BF16, QB>(a, st);
    case EPI_F32: return launch_mt<W4, EPI_F32, QB>(a, st);
    case EPI_RESID: return launch_mt<W4, EPI_RESID, QB>(a, st);
    case EPI_GLU: return launch_mt<W4, EPI_GLU, QB>(a, st);
    case EPI_QKV: return launch_mt<W4, EPI_QKV, QB>(a, st);
  }
  return fail(SUB_EINVAL, "bad gemv epilogue");
}

static int32_t launch_bf16_or_tma(const GemvArgs& a, int epi, cudaStream_t st) {
  bool done = false;
  SUB_TRY(launch_gemv_tma(a, false, epi, st, &done));
  if (done) return SUB_OK;
  return launch_epi<false, 4>(a, epi, st);
}

int32_t launch_gemv(const GemvArgs& a, bool is_w4, int epi, cudaStream_t st) {
  SUB_CHECK_ARG(a.M >= 1 && a.M <= 16, "gemv: M must be in [1, 16]");
  SUB_CHECK_ARG(a.K % 8 == 0 && a.ldx % 8 == 0, "gemv: K and ldx must be multiples of 8");
  SUB_CHECK_ARG(a.n_seg >= 1 && a.n_seg <= 4, "gemv: 1..4 segments");
  SUB_CHECK_ARG(aligned16(a.X), "gemv: X must be 16-byte aligned");
  if (a.n_seg > 1 || epi == EPI_GLU)
    for (int i = 0; i < a.n_seg; ++i) {
      const int start = i ? a.seg_end[i - 1] : 0;
      SUB_CHECK_ARG((a.seg_end[i] - start) % 16 == 0, "gemv: segments must be multiples of 16 rows");
    }
  if (epi == EPI_QKV) {
    const QkvOut& q = a.qkv;
    SUB_CHECK_ARG(a.n_seg == 3 && q.head_dim % 16 == 0 && q.head_dim >= 16, "gemv: bad q/k/v layout");
    SUB_CHECK_ARG(a.seg_end[0] == q.n_heads_q * q.head_dim &&
                      a.seg_end[1] == (q.n_heads_q + q.n_heads_kv) * q.head_dim &&
                      a.seg_end[2] == (q.n_heads_q + 2 * q.n_heads_kv) * q.head_dim &&
                      a.N == a.seg_end[2],
                  "gemv: q/k/v segment sizes");
  }
  if (epi == EPI_RESID && a.norm.xn)
    SUB_CHECK_ARG(a.norm.partial && a.norm.gain && a.ldy == a.N && a.n_seg == 1,
                  "gemv: norm epilogue needs partial, gain, one segment and ldy == N");
  const int bits = code_bits(a);
  SUB_CHECK_ARG(!is_w4 || bits == 2 || bits == 3 || bits == 4, "gemv: code bits must be 2, 3 or 4");
  if (!is_w4) return launch_bf16_or_tma(a, epi, st);
  bool done = false;
  SUB_TRY(launch_gemv_tma(a, true, epi, st, &done));
  if (done) return SUB_OK;
  if (bits == 2) return launch_epi<true, 2>(a, epi, st);
  if (bits == 3) return launch_epi<true, 3>(a, epi, st);
  return launch_epi<true, 4>(a, epi, st);
}

}  // namespace sub
