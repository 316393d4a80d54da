// Warp-level GEMV kernels (bf16 and int4 weights), see gemv.cuh.
#include "gemv.cuh"

namespace sub {

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

template <bool W4, int MT, int RT, int WK, int EPI, int U>
__global__ void __launch_bounds__(WK * 32)
gemv_kernel(GemvArgs a) {
  constexpr bool GLU = (EPI == EPI_GLU);
  constexpr int NT = GLU ? 2 * RT : RT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tig = lane & 3;
  const int n0 = blockIdx.x * (16 * RT);
  const int K = a.K;

  // ---- per-tile row pointers (two rows per lane: g and g+8) ----
  const char* rp0[NT];
  const char* rp1[NT];
  const uint16_t* sp0[NT];
  const uint16_t* sp1[NT];
  const uint16_t* zp0[NT];
  const uint16_t* zp1[NT];
  const int G = (K + 63) / 64;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int vrow = n0 + 16 * (t % RT);
    int seg = GLU ? (t / RT) : 0;
    int seg_start = 0;
    if (!GLU) {
#pragma unroll
      for (int i = 0; i < 3; ++i)
        if (seg < a.n_seg - 1 && vrow >= a.seg_end[seg]) { seg_start = a.seg_end[seg]; ++seg; }
    }
    const int seg_rows = GLU ? a.N : a.seg_end[seg] - seg_start;
    int r0 = vrow - (GLU ? 0 : seg_start) + g;
    int r1 = r0 + 8;
    r0 = min(r0, seg_rows - 1);
    r1 = min(r1, seg_rows - 1);
    if (W4) {
      const char* base = reinterpret_cast<const char*>(a.W[seg]);
      rp0[t] = base + (int64_t)r0 * G * 32 + tig * 8;
      rp1[t] = base + (int64_t)r1 * G * 32 + tig * 8;
      sp0[t] = a.S[seg] + (int64_t)r0 * G;
      sp1[t] = a.S[seg] + (int64_t)r1 * G;
      zp0[t] = a.Z[seg] + (int64_t)r0 * G;
      zp1[t] = a.Z[seg] + (int64_t)r1 * G;
    } else {
      const char* base = reinterpret_cast<const char*>(a.W[seg]);
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
    const int steps = (K + 31) / 32;
    const int per = (steps + WK - 1) / WK;
    const int s_begin = warp * per, s_end = min(steps, s_begin + per);
    for (int s = s_begin; s < s_end; s += U) {
      uint4 w0[U][NT], w1[U][NT], xv[U][MT];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = (s + u) * 32 + tig * 8;
        const bool ok = (s + u < s_end) && (k < K);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          w0[u][t] = ok ? ldg_nc_v4(rp0[t] + (int64_t)(s + u) * 64) : make_uint4(0, 0, 0, 0);
          w1[u][t] = ok ? ldg_nc_v4(rp1[t] + (int64_t)(s + u) * 64) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          xv[u][mt] = (ok && xok[mt]) ? __ldg(reinterpret_cast<const uint4*>(xp[mt] + k))
                                      : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t A0[4] = {w0[u][t].x, w1[u][t].x, w0[u][t].y, w1[u][t].y};
            const uint32_t A1[4] = {w0[u][t].z, w1[u][t].z, w0[u][t].w, w1[u][t].w};
            mma_bf16_16816(acc[t][mt], A0, xv[u][mt].x, xv[u][mt].y);
            mma_bf16_16816(acc[t][mt], A1, xv[u][mt].z, xv[u][mt].w);
          }
    }
  } else {
    // ------------------------------------------------ int4 weights ----
    const int per = (G + WK - 1) / WK;
    const int g_begin = warp * per, g_end = min(G, g_begin + per);
    const uint32_t ONES = 0x3f803f80u;
    const uint32_t ONES_A[4] = {ONES, ONES, ONES, ONES};
    for (int gi0 = g_begin; gi0 < g_end; gi0 += U) {
      uint2 q0[U][NT], q1[U][NT];
      uint16_t s0[U][NT], s1[U][NT], z0[U][NT], z1[U][NT];
      uint4 xa[U][MT], xb[U][MT];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int gi = gi0 + u;
        const bool ok = gi < g_end;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          q0[u][t] = ok ? ldg_nc_v2(rp0[t] + (int64_t)gi * 32) : make_uint2(0, 0);
          q1[u][t] = ok ? ldg_nc_v2(rp1[t] + (int64_t)gi * 32) : make_uint2(0, 0);
          s0[u][t] = ok ? __ldg(sp0[t] + gi) : 0;
          s1[u][t] = ok ? __ldg(sp1[t] + gi) : 0;
          z0[u][t] = ok ? __ldg(zp0[t] + gi) : 0;
          z1[u][t] = ok ? __ldg(zp1[t] + gi) : 0;
        }
        const int k = gi * 64 + tig * 16;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          xa[u][mt] = (ok && xok[mt] && k < K) ? __ldg(reinterpret_cast<const uint4*>(xp[mt] + k))
                                               : make_uint4(0, 0, 0, 0);
          xb[u][mt] = (ok && xok[mt] && k + 8 < K)
                          ? __ldg(reinterpret_cast<const uint4*>(xp[mt] + k + 8))
                          : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        // B fragments: pairs (k, k+4) to match the nibble pairs of one word
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
          // nibble pairs (n_i, n_{i+4}) of each word -> bf16x2 (128 + q)
          uint32_t A[4][4];
          {
            const uint32_t a0 = q0[u][t].x, a1 = q0[u][t].y;   // row g: words 0, 1
            const uint32_t c0 = q1[u][t].x, c1 = q1[u][t].y;   // row g+8
            const uint32_t NIB = 0x000f000fu, E = 0x43004300u;
            // mma i reads word i/2 of each row: nibble pairs (0,4),(1,5) for even
            // i and (2,6),(3,7) for odd i; the B fragments pair K the same way
            A[0][0] = (a0 & NIB) | E;         A[0][2] = ((a0 >> 4) & NIB) | E;
            A[0][1] = (c0 & NIB) | E;         A[0][3] = ((c0 >> 4) & NIB) | E;
            A[1][0] = ((a0 >> 8) & NIB) | E;  A[1][2] = ((a0 >> 12) & NIB) | E;
            A[1][1] = ((c0 >> 8) & NIB) | E;  A[1][3] = ((c0 >> 12) & NIB) | E;
            A[2][0] = (a1 & NIB) | E;         A[2][2] = ((a1 >> 4) & NIB) | E;
            A[2][1] = (c1 & NIB) | E;         A[2][3] = ((c1 >> 4) & NIB) | E;
            A[3][0] = ((a1 >> 8) & NIB) | E;  A[3][2] = ((a1 >> 12) & NIB) | E;
            A[3][1] = ((c1 >> 8) & NIB) | E;  A[3][3] = ((c1 >> 12) & NIB) | E;
          }
          const float sr0 = bf16_bits_to_f32(s0[u][t]), sr1 = bf16_bits_to_f32(s1[u][t]);
          const float zr0 = 128.0f + bf16_bits_to_f32(z0[u][t]);
          const float zr1 = 128.0f + bf16_bits_to_f32(z1[u][t]);
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
      }
    }
  }

  // ---- cross-warp reduction in a fixed order, then the epilogue ----
  static_assert(WK >= 2, "the epilogue reads partial sums through shared memory");
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
  constexpr int OUT_ELEMS = RT * MT * 4 * 32;
  for (int e = threadIdx.x; e < OUT_ELEMS; e += WK * 32) {
    // e = ((t * MT + mt) * 4 + j) * 32 + ln, t < RT
    const int ln = e & 31;
    const int j = (e >> 5) & 3;
    const int mt = (e >> 7) % MT;
    const int t = (e >> 7) / MT;
    float v = 0.f, vu = 0.f;
#pragma unroll
    for (int w = 0; w < WK; ++w) v += red[w * PER_WARP + e];
    if constexpr (GLU) {
      const int eu = e + RT * MT * 4 * 32;   // same element of the 'up' tile t + RT
#pragma unroll
      for (int w = 0; w < WK; ++w) vu += red[w * PER_WARP + eu];
    }
    const int gg = ln >> 2, tg = ln & 3;
    const int row = n0 + 16 * t + gg + ((j & 2) ? 8 : 0);
    const int tok = mt * 8 + 2 * tg + (j & 1);
    if (row >= a.N || tok >= a.M) continue;
    const int64_t o = (int64_t)tok * a.ldy + row;
    if constexpr (EPI == EPI_BF16) {
      reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(v);
    } else if constexpr (EPI == EPI_F32) {
      reinterpret_cast<float*>(a.Y)[o] = v;
    } else if constexpr (EPI == EPI_RESID) {
      reinterpret_cast<float*>(a.Y)[o] += v;
    } else {
      reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(silu_f(v) * vu);
    }
  }
}

template <bool W4, int MT, int RT, int WK, int EPI>
static int32_t launch_cfg(const GemvArgs& a, cudaStream_t st) {
  constexpr int U = W4 ? 4 : 4;
  const int blocks = (a.N + 16 * RT - 1) / (16 * RT);
  gemv_kernel<W4, MT, RT, WK, EPI, U><<<blocks, WK * 32, 0, st>>>(a);
  return check_launch("gemv");
}

template <bool W4, int MT, int EPI>
static int32_t launch_rt(const GemvArgs& a, cudaStream_t st) {
  // Segments must not straddle a CTA's rows: two row tiles per CTA when every
  // segment is a multiple of 32 rows and the grid stays wide enough.
  bool rt2 = (EPI != EPI_GLU) && a.N >= 32 * 152;
  for (int i = 0; i < a.n_seg; ++i) {
    const int start = i ? a.seg_end[i - 1] : 0;
    if ((a.seg_end[i] - start) % 32) rt2 = false;
  }
  if (rt2) return launch_cfg<W4, MT, 2, 4, EPI>(a, st);
  return launch_cfg<W4, MT, 1, 4, EPI>(a, st);
}

template <bool W4, int EPI>
static int32_t launch_mt(const GemvArgs& a, cudaStream_t st) {
  if (a.M <= 8) return launch_rt<W4, 1, EPI>(a, st);
  return launch_rt<W4, 2, EPI>(a, st);
}

template <bool W4>
static int32_t launch_epi(const GemvArgs& a, int epi, cudaStream_t st) {
  switch (epi) {
    case EPI_BF16: return launch_mt<W4, EPI_BF16>(a, st);
    case EPI_F32: return launch_mt<W4, EPI_F32>(a, st);
    case EPI_RESID: return launch_mt<W4, EPI_RESID>(a, st);
    case EPI_GLU: return launch_mt<W4, EPI_GLU>(a, st);
  }
  return fail(SUB_EINVAL, "bad gemv epilogue");
}

int32_t launch_gemv(const GemvArgs& a, bool is_w4, int epi, cudaStream_t st) {
  SUB_CHECK_ARG(a.M >= 1 && a.M <= 16, "gemv: M must be in [1, 16]");
  SUB_CHECK_ARG(a.K % 8 == 0 && a.ldx % 8 == 0, "gemv: K and ldx must be multiples of 8");
  SUB_CHECK_ARG(a.n_seg >= 1 && a.n_seg <= 4, "gemv: 1..4 segments");
  if (a.n_seg > 1 || epi == EPI_GLU)
    for (int i = 0; i < a.n_seg; ++i) {
      const int start = i ? a.seg_end[i - 1] : 0;
      SUB_CHECK_ARG((a.seg_end[i] - start) % 16 == 0, "gemv: segments must be multiples of 16 rows");
    }
  return is_w4 ? launch_epi<true>(a, epi, st) : launch_epi<false>(a, epi, st);
}

}  // namespace sub
