// Draft-shaped GEMV (M <= 16 activation rows) streamed through shared memory
// by the Tensor Memory Accelerator.
//
// Y[m, n] = sum_k X[m, k] W[n, k], the same products and epilogues as the
// register-streamed kernel in gemv.cu, for bf16 weights or 4-, 3- or 2-bit
// substitutes (W = (q - z) * s per 64-column group).  A small M leaves the product bound
// by the weight stream, and the number of weight bytes in flight per SM is
// what decides the bandwidth reached.  Here the bytes in flight live in a
// shared-memory ring instead of registers:
//
//   * one producer warp issues 2-D TMA copies (cp.async.bulk.tensor) of each
//     stage -- a 128-row block of weights (bf16 rows, or packed nibbles plus
//     their scales and zeros) over KC columns, and the matching X columns --
//     into a ring of S stages, each guarded by a full and an empty mbarrier;
//   * eight consumer warps each own a 16-row tile of the block and run
//     mma.sync m16n8k16 (swap-AB: W is the A operand, X the B operand)
//     straight from the swizzled stages, then release the stage;
//   * 2- and 3-bit codes take the same path: a stage's 8 groups are 128
//     bytes of a row (2-bit) or 192 (3-bit: a 128-byte box and a 64-byte
//     one with the 64-byte swizzle); 2-bit codes go straight to the operand
//     pairs after one byte permute per word, 3-bit codes are first spread
//     into the int4 word layout;
//   * with int4 weights two more warps (even and odd groups) form each
//     stage's per-group activation sums Sx (an mma with an all-ones A
//     operand) and, for one token tile, the activation B fragments in lane
//     order, once for all eight tiles, and hand them over in the stage, so
//     the consumers only unpack, multiply and fold.
//
// The weights of the first stages are requested before the wait on the
// producing kernel (programmatic dependent launch); only X waits for it.
//
// Work balance (stream-K): the (block, stage) units of the whole product are
// cut into one contiguous range per CTA, one CTA per SM.  A block finished by
// a single CTA goes straight to the epilogue; a block shared by several CTAs
// is summed by the last of them to arrive, in CTA order (deterministic).
//
// Shared-memory banks: the TMA 128-byte swizzle stores 16-byte chunk c of a
// 128-byte row r at chunk position c ^ (r & 7).  The fragment row g of a lane
// reads smem row base + pi(g), with pi chosen so that the lanes of one shared
// load phase hit eight distinct chunk positions: pi = (0,4,1,5,2,6,3,7) for
// bf16 (16-byte reads, two rows per phase) and pi = (0,2,4,6,1,3,5,7) for int4
// (8-byte reads, four rows per phase).  bf16 activations use the same pi on
// their token rows.  The epilogue maps fragment rows and tokens back through pi.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <mutex>
#include "gemv.cuh"
#include "tma.cuh"

namespace sub {

namespace {

using namespace tmah;

constexpr int NCW = 8;                  // consumer warps; one 16-row tile each
constexpr int NTHR = (NCW + 1) * 32;    // plus the producer warp
constexpr int NTHR_W4 = NTHR + 64;      // plus two group-sum warps (int4)
constexpr int BR = NCW * 16;            // rows of a block
constexpr int SMEM_LIMIT = 220 * 1024;  // dynamic shared memory of one CTA (1 per SM)
constexpr int MAX_STAGES = 6;

__device__ unsigned int g_tma_timeouts;  // waits that ran out (never expected)

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Bounded wait: one that runs out is counted (sub_pipeline_timeouts) and the
// kernel goes on with wrong numbers instead of hanging.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity) {
  if (!mbar_wait_polls(bar, parity, 1u << 20)) atomicAdd(&g_tma_timeouts, 1u);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short r;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
  return r;
}

// Shared address of byte `off` of smem row r of a stage's 2/3-bit codes:
// bytes 0..127 in the 128-byte-swizzled box (16-byte chunk c of row r at
// c ^ (r & 7)), bytes 128..191 in the 64-byte-swizzled box (chunk c of its
// 64-byte row r at c ^ ((r >> 1) & 3)).
__device__ __forceinline__ uint32_t code_addr(uint32_t box128, uint32_t box64, int r, int off) {
  return off < 128 ? box128 + r * 128 + ((((off >> 4) ^ r) & 7) << 4) + (off & 15)
                   : box64 + r * 64 + (((((off - 128) >> 4) ^ (r >> 1)) & 3) << 4) + (off & 15);
}

// One lane's 16 codes of stage group gs (elements 16 tig .. 16 tig + 15 of
// the group) from smem row r, in the int4 word layout (the same words the
// register-streamed kernel forms from global memory).
template <int QB>
__device__ __forceinline__ uint2 stage_codes(uint32_t box128, uint32_t box64, int r, int gs, int tig) {
  const int g0 = gs * 8 * QB;
  const uint32_t w = lds32(code_addr(box128, box64, r, g0 + tig * 4));
  uint2 q = make_uint2(spread2(w), spread2(w >> 16));
  if constexpr (QB == 3) {
    const uint32_t h = lds16(code_addr(box128, box64, r, g0 + 16 + tig * 2));
    q.x |= spread1(h) << 2;
    q.y |= spread1(h >> 8) << 2;
  }
  return q;
}

}  // namespace

struct alignas(64) TmaMaps {
  CUtensorMap w[3];   // bf16 weights, or packed int4 codes, per segment
  CUtensorMap s[3];   // int4 scales per segment
  CUtensorMap z[3];   // int4 zeros per segment
  CUtensorMap w64[3]; // 3-bit codes: bytes 128..191 of a stage's 192 per row
  CUtensorMap x;      // activations [M, K] viewed as [K/64][M][64]: one box per stage
};

struct TmaPlan {
  int n_blocks;       // 128-row blocks (GLU: 64 gate + 64 up rows)
  int blk_end[3];     // cumulative blocks per segment
  int s_blk;          // stages per block (over the whole K)
  int total;          // n_blocks * s_blk
  int maxc;           // partial slots per block
  int n_maps;         // weight segments with a tensor map
};

template <bool W4, int MT, int QB = 4>
struct TmaGeom {
  static constexpr int KC = W4 ? 512 : 128;              // K columns per stage
  // weight boxes per stage, 128 B wide: bf16 and 4-bit two, 2-bit one, 3-bit
  // one plus a 64-byte box (W64)
  static constexpr int WBOXES = W4 && QB < 4 ? 1 : 2;
  static constexpr int WBOX = BR * 128;                  // bytes of one weight box (all rows)
  static constexpr int W64 = W4 && QB == 3 ? BR * 64 : 0;
  static constexpr int SZBOX = W4 ? BR * 16 : 0;         // scales (or zeros) of 8 groups
  static constexpr int XBOXES = KC / 64;                 // activation boxes (64 columns each)
  static constexpr int XBOX = MT * 8 * 128;              // bytes of one activation box
  static constexpr int W_OFF = 0;
  static constexpr int W64_OFF = WBOXES * WBOX;          // 1024-byte aligned (swizzle span)
  static constexpr int S_OFF = W64_OFF + W64;
  static constexpr int Z_OFF = S_OFF + SZBOX;
  static constexpr int X_OFF = (Z_OFF + SZBOX + 1023) / 1024 * 1024;
  static constexpr int SX_OFF = X_OFF + XBOXES * XBOX;   // int4: Sx [8 groups][MT * 8 tokens] fp32
  static constexpr int SXB = W4 ? 8 * MT * 8 * 4 : 0;
  // int4, one token tile: the stage's activation B fragments in lane order,
  // [8 groups][2 halves][32 lanes][16 bytes], formed once by the group-sum warp
  static constexpr bool XFRAG = W4 && MT == 1;
  static constexpr int XF_OFF = SX_OFF + SXB;
  static constexpr int XFB = XFRAG ? 8 * 2 * 32 * 16 : 0;
  static constexpr int STAGE = (XF_OFF + XFB + 1023) / 1024 * 1024;
  static constexpr int TX = WBOXES * WBOX + W64 + 2 * SZBOX + XBOXES * XBOX;   // bytes per stage
  // + flag (16 floats), row scales (one per activation row)
  static constexpr int EPI_FLOATS = 4 * MT * 128 + NCW * 16 + 16 + (MT > 2 ? MT * 8 : 16);
  // alignment slack, ring, barriers and epilogue buffers within the limit
  static constexpr int STAGES =
      std::min(MAX_STAGES, (SMEM_LIMIT - 1024 - 3 * MAX_STAGES * 8 - EPI_FLOATS * 4) / STAGE);
  static constexpr int SMEM = 1024 + STAGES * STAGE + 3 * STAGES * 8 + EPI_FLOATS * 4;
  static_assert(STAGES >= 3 && SMEM <= SMEM_LIMIT, "TMA GEMV ring does not fit");
};

template <bool W4, int MT, int EPI, int QB = 4>
__global__ void __launch_bounds__(W4 ? NTHR_W4 : NTHR, 1)
gemv_tma_kernel(const __grid_constant__ TmaMaps maps, const GemvArgs a, const TmaPlan pl) {
  using Geo = TmaGeom<W4, MT, QB>;
  constexpr int S = Geo::STAGES;
  constexpr bool GLU = EPI == EPI_GLU;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled boxes
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t bars = base + S * Geo::STAGE;          // full[S], empty[S], sums[S]
  float* const epi = reinterpret_cast<float*>(base_ptr + S * Geo::STAGE + 3 * S * 8);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto sx_bar = [&](int s) { return bars + 8u * (2 * S + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = gridDim.x, c = blockIdx.x;
  const int u0 = (int)((int64_t)c * pl.total / P), u1 = (int)((int64_t)(c + 1) * pl.total / P);

  if (warp == NCW && lane == 0) {   // descriptors into the TMA unit's cache early
    for (int t = 0; t < pl.n_maps; ++t) {
      tma_prefetch_desc(&maps.w[t]);
      if (W4 && QB == 3) tma_prefetch_desc(&maps.w64[t]);
      if (W4) {
        tma_prefetch_desc(&maps.s[t]);
        tma_prefetch_desc(&maps.z[t]);
      }
    }
    tma_prefetch_desc(&maps.x);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), NCW);
      mbar_init(sx_bar(s), 2);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // block -> (segment, first row of the segment's block)
  auto block_seg = [&](int b, int* seg, int* r0) {
    int s = 0;
    while (s < 2 && b >= pl.blk_end[s]) ++s;
    *seg = s;
    *r0 = (b - (s ? pl.blk_end[s - 1] : 0)) * (GLU ? BR / 2 : BR);
  };

  // ================================================================ producer
  if (warp == NCW) {
    if (lane == 0) {
      auto issue = [&](int u, bool weights, bool acts) {
        const int i = u - u0, s = i % S;
        const int b = u / pl.s_blk, kst = u % pl.s_blk;
        int seg, r0;
        block_seg(b, &seg, &r0);
        const uint32_t st = base + s * Geo::STAGE, fb = full_bar(s);
        if (weights) {
          mbar_expect_tx(fb, Geo::TX);
          if constexpr (W4) {
            const int gx = kst * (Geo::KC / 64);        // first group of the stage
            for (int h = 0; h < (GLU ? 2 : 1); ++h) {
              const int sg = GLU ? h : seg, rows = GLU ? BR / 2 : BR;
              const uint32_t ro = h * rows * 128;       // row offset inside a box (bytes)
              if constexpr (QB == 4) {
                for (int j = 0; j < Geo::WBOXES; ++j)
                  tma_load_2d(st + Geo::W_OFF + j * Geo::WBOX + ro, &maps.w[sg], (gx + 4 * j) * 32, r0, fb);
              } else {
                // the stage's 8 groups of 8 QB bytes: 128 bytes (2-bit), or
                // 128 + 64 bytes (3-bit); x in bytes, a multiple of 16
                tma_load_2d(st + Geo::W_OFF + ro, &maps.w[sg], gx * 8 * QB, r0, fb);
                if constexpr (QB == 3)
                  tma_load_2d(st + Geo::W64_OFF + h * rows * 64, &maps.w64[sg], gx * 24 + 128, r0, fb);
              }
              tma_load_2d(st + Geo::S_OFF + h * rows * 16, &maps.s[sg], gx, r0, fb);
              tma_load_2d(st + Geo::Z_OFF + h * rows * 16, &maps.z[sg], gx, r0, fb);
            }
          } else {
            const int kx = kst * Geo::KC;
            for (int h = 0; h < (GLU ? 2 : 1); ++h) {
              const int sg = GLU ? h : seg, rows = GLU ? BR / 2 : BR;
              const uint32_t ro = h * rows * 128;
              for (int j = 0; j < Geo::WBOXES; ++j)
                tma_load_2d(st + Geo::W_OFF + j * Geo::WBOX + ro, &maps.w[sg], kx + 64 * j, r0, fb);
            }
          }
        }
        // the stage's XBOXES 64-column slices of X, one after another, in one copy
        if (acts) tma_load_3d(st + Geo::X_OFF, &maps.x, 0, 0, kst * Geo::XBOXES, fb);
      };
      const int npre = std::min(S, u1 - u0);
      for (int u = u0; u < u0 + npre; ++u) issue(u, true, false);   // weights before the wait
      pdl_wait();
      for (int u = u0; u < u0 + npre; ++u) issue(u, false, true);
      for (int u = u0 + npre; u < u1; ++u) {
        const int i = u - u0;
        mbar_wait(empty_bar(i % S), ((i / S) - 1) & 1);
        issue(u, true, true);
      }
    }
    __syncwarp();   // lanes 1..31 signal only once lane 0 has passed the wait
    pdl_trigger();
    return;
  }

  const int g = lane >> 2, tig = lane & 3;
  const uint32_t ONES = 0x3f803f80u;   // bf16x2 (1, 1)
  const uint32_t ONES_A[4] = {ONES, ONES, ONES, ONES};
  // B fragments of the 16 columns of 64-column activation box xbox that lane
  // (g, tig) holds for token tile mt: columns (k, k + 4) paired, k-step kk
  auto x_frags = [&](uint32_t xbox, int mt, uint32_t (&bfr)[4][2]) {
    const int xr = mt * 8 + g;
    const uint4 xa = lds128(xbox + xr * 128 + (((2 * tig) ^ g) << 4));
    const uint4 xc = lds128(xbox + xr * 128 + (((2 * tig + 1) ^ g) << 4));
    bfr[0][0] = __byte_perm(xa.x, xa.z, 0x5410);
    bfr[0][1] = __byte_perm(xa.x, xa.z, 0x7632);
    bfr[1][0] = __byte_perm(xa.y, xa.w, 0x5410);
    bfr[1][1] = __byte_perm(xa.y, xa.w, 0x7632);
    bfr[2][0] = __byte_perm(xc.x, xc.z, 0x5410);
    bfr[2][1] = __byte_perm(xc.x, xc.z, 0x7632);
    bfr[3][0] = __byte_perm(xc.y, xc.w, 0x5410);
    bfr[3][1] = __byte_perm(xc.y, xc.w, 0x7632);
  };

  // ================================================================ group sums
  if constexpr (W4) {
    if (warp == NCW + 1 || warp == NCW + 2) {
      const int par = warp - (NCW + 1);   // this warp's groups: par, par + 2, ...
      for (int u = u0; u < u1; ++u) {
        const int i = u - u0, s = i % S;
        const uint32_t st = base + s * Geo::STAGE;
        mbar_wait(full_bar(s), (i / S) & 1);
#pragma unroll
        for (int gh = 0; gh < 4; ++gh)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int gs = 2 * gh + par;
            uint32_t bfr[4][2];
            x_frags(st + Geo::X_OFF + gs * Geo::XBOX, mt, bfr);
            if constexpr (Geo::XFRAG) {
              const uint32_t xf = st + Geo::XF_OFF + ((gs * 2) * 32 + lane) * 16;
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xf), "r"(bfr[0][0]),
                           "r"(bfr[0][1]), "r"(bfr[1][0]), "r"(bfr[1][1])
                           : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xf + 32 * 16),
                           "r"(bfr[2][0]), "r"(bfr[2][1]), "r"(bfr[3][0]), "r"(bfr[3][1])
                           : "memory");
            }
            float sx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_bf16_16816(sx, ONES_A, bfr[k][0], bfr[k][1]);
            // every row of the result is Sx; row 0 holds tokens 2 tig, 2 tig + 1
            if (g == 0)
              asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(
                               st + Geo::SX_OFF + (((gs * MT + mt) * 8 + 2 * tig) << 2)),
                           "f"(sx[0]), "f"(sx[1])
                           : "memory");
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(sx_bar(s));
      }
      pdl_trigger();
      return;
    }
  }

  // ================================================================ consumers
  pdl_wait();
  // row scales of a factored RMSNorm input, from the producer's per-tile sums
  float* const s_r = epi + 4 * MT * 128 + NCW * 16 + 16;
  if (a.xscale.partial) {
    for (int m = warp; m < a.M; m += NCW) {
      const float r = row_scale(a.xscale, m, lane);
      if (lane == 0) s_r[m] = r;
    }
    consumer_sync();
  }
  // row permutation pi of the fragment rows (and bf16 token rows)
  const int pg = W4 ? ((g & 3) * 2 + (g >> 2)) : ((g & 1) * 4 + (g >> 1));
  const int ptok_x = W4 ? g : pg;   // smem token row of B column g

  float acc[MT][4];
  int seg = 0, r0 = 0, lo = 0, hi = 0, piece_start = 0;
  for (int u = u0; u < u1; ++u) {
    const int i = u - u0, s = i % S;
    const int b = u / pl.s_blk, kst = u % pl.s_blk;
    if (u == u0 || kst == 0) {
      block_seg(b, &seg, &r0);
      piece_start = kst;
      // smem rows of this warp's tile: fragment rows g -> lo + pi(g), g + 8 -> hi + pi(g)
      lo = warp * 16;
      hi = lo + 8;
      if constexpr (EPI == EPI_QKV) {
        if (seg < 2) {
          const int D = a.qkv.head_dim, per_head = D / 16;
          lo = (warp / per_head) * D + 8 * (warp % per_head);
          hi = lo + D / 2;
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[mt][j] = 0.f;
    }
    const uint32_t st = base + s * Geo::STAGE;
    mbar_wait(W4 ? sx_bar(s) : full_bar(s), (i / S) & 1);   // sums imply the bytes landed
    const int r0s = lo + pg, r1s = hi + pg;   // smem rows; (r & 7) == pg

    if constexpr (!W4) {
      // ---------------------------------------------------- bf16 weights
#pragma unroll
      for (int j = 0; j < Geo::WBOXES; ++j) {
        const uint32_t wb = st + Geo::W_OFF + j * Geo::WBOX;
        const uint32_t xb = st + Geo::X_OFF + j * Geo::XBOX;
#pragma unroll
        for (int h = 0; h < 2; ++h) {          // two steps of 32 columns per 64-column box
          const uint32_t co = (uint32_t)(((h * 4 + tig) ^ pg) << 4);
          const uint4 w0 = lds128(wb + r0s * 128 + co);
          const uint4 w1 = lds128(wb + r1s * 128 + co);
          const uint32_t A0[4] = {w0.x, w1.x, w0.y, w1.y};
          const uint32_t A1[4] = {w0.z, w1.z, w0.w, w1.w};
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint4 xv = lds128(xb + (mt * 8 + ptok_x) * 128 + co);
            mma_bf16_16816(acc[mt], A0, xv.x, xv.y);
            mma_bf16_16816(acc[mt], A1, xv.z, xv.w);
          }
        }
      }
    } else {
      // ---------------------------------------------------- int4 weights
      // scales and zeros of the stage's 8 groups for rows r0s, r1s
      const uint4 sv0 = lds128(st + Geo::S_OFF + r0s * 16), sv1 = lds128(st + Geo::S_OFF + r1s * 16);
      const uint4 zv0 = lds128(st + Geo::Z_OFF + r0s * 16), zv1 = lds128(st + Geo::Z_OFF + r1s * 16);
      const uint32_t sw0[4] = {sv0.x, sv0.y, sv0.z, sv0.w}, sw1[4] = {sv1.x, sv1.y, sv1.z, sv1.w};
      const uint32_t zw0[4] = {zv0.x, zv0.y, zv0.z, zv0.w}, zw1[4] = {zv1.x, zv1.y, zv1.z, zv1.w};
#pragma unroll
      for (int gs = 0; gs < 8; ++gs) {
        // int4 layout words (code i of a run of 8 at bits 4i), or at 2 bits
        // byte pairs (codes i and i + 4 of a run of 8 at bits 2i and 16 + 2i)
        uint2 q0, q1;
        if constexpr (QB == 4) {
          const int j = gs >> 2, gq = gs & 3;
          const uint32_t qb = st + Geo::W_OFF + j * Geo::WBOX;
          const uint32_t qo = (uint32_t)((((2 * gq + (tig >> 1)) ^ pg) << 4) + (tig & 1) * 8);
          q0 = lds64(qb + r0s * 128 + qo);
          q1 = lds64(qb + r1s * 128 + qo);
        } else if constexpr (QB == 2) {
          const int off = gs * 16 + tig * 4;
          const uint32_t w0 = lds32(code_addr(st + Geo::W_OFF, st + Geo::W_OFF, r0s, off));
          const uint32_t w1 = lds32(code_addr(st + Geo::W_OFF, st + Geo::W_OFF, r1s, off));
          q0 = make_uint2(__byte_perm(w0, 0u, 0x4140), __byte_perm(w0, 0u, 0x4342));
          q1 = make_uint2(__byte_perm(w1, 0u, 0x4140), __byte_perm(w1, 0u, 0x4342));
        } else {
          q0 = stage_codes<QB>(st + Geo::W_OFF, st + Geo::W64_OFF, r0s, gs, tig);
          q1 = stage_codes<QB>(st + Geo::W_OFF, st + Geo::W64_OFF, r1s, gs, tig);
        }
        const uint32_t xbox = st + Geo::X_OFF + gs * Geo::XBOX;
        // up to two token tiles: every tile's B fragments and sums up front;
        // four: one tile at a time, after the unpack (registers)
        constexpr int MTU = MT > 2 ? 1 : MT;
        uint32_t bfr[MTU][4][2];
        float sx[MTU][2];
#pragma unroll
        for (int mt = 0; mt < (MT > 2 ? 0 : MT); ++mt) {
          if constexpr (Geo::XFRAG) {
            const uint32_t xf = st + Geo::XF_OFF + ((gs * 2) * 32 + lane) * 16;
            const uint4 f0 = lds128(xf), f1 = lds128(xf + 32 * 16);
            bfr[mt][0][0] = f0.x;
            bfr[mt][0][1] = f0.y;
            bfr[mt][1][0] = f0.z;
            bfr[mt][1][1] = f0.w;
            bfr[mt][2][0] = f1.x;
            bfr[mt][2][1] = f1.y;
            bfr[mt][3][0] = f1.z;
            bfr[mt][3][1] = f1.w;
          } else {
            x_frags(xbox, mt, bfr[mt]);
          }
          asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                       : "=f"(sx[mt][0]), "=f"(sx[mt][1])
                       : "r"(st + Geo::SX_OFF + (((gs * MT + mt) * 8 + 2 * tig) << 2)));
        }
        const uint32_t a0s = (gs & 1) ? (sw0[gs >> 1] >> 16) : (sw0[gs >> 1] & 0xffffu);
        const uint32_t a1s = (gs & 1) ? (sw1[gs >> 1] >> 16) : (sw1[gs >> 1] & 0xffffu);
        const uint32_t b0z = (gs & 1) ? (zw0[gs >> 1] >> 16) : (zw0[gs >> 1] & 0xffffu);
        const uint32_t b1z = (gs & 1) ? (zw1[gs >> 1] >> 16) : (zw1[gs >> 1] & 0xffffu);
        const float sr0 = __uint_as_float(a0s << 16), sr1 = __uint_as_float(a1s << 16);
        const float zr0 = 128.0f + __uint_as_float(b0z << 16);
        const float zr1 = 128.0f + __uint_as_float(b1z << 16);
        // code pairs (q_i, q_{i+4}) of each word -> bf16x2 (128 + q), K paired
        // (k, k + 4) on both operands; SH bits per code step
        uint32_t A[4][4];
        {
          constexpr int SH = QB == 2 ? 2 : 4;
          constexpr uint32_t MK = QB == 2 ? 0x00030003u : 0x000f000fu;
          const uint32_t E = 0x43004300u;
          const uint32_t a0 = q0.x, a1 = q0.y, c0 = q1.x, c1 = q1.y;
          A[0][0] = (a0 & MK) | E;               A[0][2] = ((a0 >> SH) & MK) | E;
          A[0][1] = (c0 & MK) | E;               A[0][3] = ((c0 >> SH) & MK) | E;
          A[1][0] = ((a0 >> (2 * SH)) & MK) | E; A[1][2] = ((a0 >> (3 * SH)) & MK) | E;
          A[1][1] = ((c0 >> (2 * SH)) & MK) | E; A[1][3] = ((c0 >> (3 * SH)) & MK) | E;
          A[2][0] = (a1 & MK) | E;               A[2][2] = ((a1 >> SH) & MK) | E;
          A[2][1] = (c1 & MK) | E;               A[2][3] = ((c1 >> SH) & MK) | E;
          A[3][0] = ((a1 >> (2 * SH)) & MK) | E; A[3][2] = ((a1 >> (3 * SH)) & MK) | E;
          A[3][1] = ((c1 >> (2 * SH)) & MK) | E; A[3][3] = ((c1 >> (3 * SH)) & MK) | E;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int mu = MT > 2 ? 0 : mt;   // register slot of this tile's operands
          if constexpr (MT > 2) {
            x_frags(xbox, mt, bfr[0]);
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                         : "=f"(sx[0][0]), "=f"(sx[0][1])
                         : "r"(st + Geo::SX_OFF + (((gs * MT + mt) * 8 + 2 * tig) << 2)));
          }
          float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t Ak[4] = {A[k][0], A[k][1], A[k][2], A[k][3]};
            mma_bf16_16816(p, Ak, bfr[mu][k][0], bfr[mu][k][1]);
          }
          acc[mt][0] = fmaf(sr0, fmaf(-zr0, sx[mu][0], p[0]), acc[mt][0]);
          acc[mt][1] = fmaf(sr0, fmaf(-zr0, sx[mu][1], p[1]), acc[mt][1]);
          acc[mt][2] = fmaf(sr1, fmaf(-zr1, sx[mu][0], p[2]), acc[mt][2]);
          acc[mt][3] = fmaf(sr1, fmaf(-zr1, sx[mu][1], p[3]), acc[mt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(s));

    // ---------------------------------------------------- end of a block piece
    if (kst != pl.s_blk - 1 && u != u1 - 1) continue;
    if (u == u1 - 1) pdl_trigger();
    const bool whole = piece_start == 0 && kst == pl.s_blk - 1;
    // fragment element j of token tile mt: smem row (j & 2 ? hi : lo) + pg,
    // B column 2 tig + (j & 1) -> token mt * 8 + tokmap(column)
    auto token_of = [&](int mt, int j) {
      const int col = 2 * tig + (j & 1);
      const int pc = W4 ? col : ((col & 1) * 4 + (col >> 1));
      return mt * 8 + pc;
    };
    const int seg_rows = GLU ? a.N : a.seg_end[seg] - (seg ? a.seg_end[seg - 1] : 0);
    const int seg_start = GLU ? 0 : (seg ? a.seg_end[seg - 1] : 0);
    // residual: the old values of the lane's elements, loaded before the
    // pieces are exchanged so that their latency hides behind it (only the
    // CTA that finishes the block writes these rows, and only after this)
    float yold[MT][4];
    if constexpr (EPI == EPI_RESID) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tok = token_of(mt, j);
          const int rs = r0 + ((j & 2) ? hi : lo) + pg;
          yold[mt][j] = (tok < a.M && rs < seg_rows)
                            ? __ldcg(reinterpret_cast<const float*>(a.Y) + (int64_t)tok * a.ldy +
                                     seg_start + rs)
                            : 0.f;
        }
    }
    float tot[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) tot[mt][j] = acc[mt][j];
    if (!whole) {
      // several CTAs share this block: park the piece, the last to arrive adds all
      const int64_t T = pl.total;
      const int c_first = (int)((((int64_t)b * pl.s_blk + 1) * P - 1) / T);
      const int c_last = (int)((((int64_t)(b + 1) * pl.s_blk) * P - 1) / T);
      const int n_c = c_last - c_first + 1;
      constexpr int PER = NCW * MT * 128;
      float* slots = a.split_part + (size_t)b * pl.maxc * PER;
      float* mine = slots + (size_t)(c - c_first) * PER + warp * MT * 128;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) __stcg(mine + mt * 128 + j * 32 + lane, acc[mt][j]);
      unsigned int* flag = reinterpret_cast<unsigned int*>(epi + 4 * MT * 128 + NCW * 16);
      consumer_sync();
      if (threadIdx.x == 0) {
        // release this CTA's piece, acquire the others' (one acq_rel atomic)
        unsigned int old;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(a.split_cnt + b)
                     : "memory");
        *flag = old == (unsigned)n_c - 1 ? 1u : 0u;
      }
      consumer_sync();
      if (!*flag) continue;
      // sum the pieces in CTA order; YY pieces' loads in flight per round
      // (one load at a time would put n_c round trips on the kernel's tail)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[mt][j] = 0.f;
      const float* mine0 = slots + warp * MT * 128 + lane;
      constexpr int YY = MT > 2 ? 2 : 8;   // pieces per round (registers at 4 tiles)
      for (int y0 = 0; y0 < n_c; y0 += YY) {
        float t[YY][MT][4];
#pragma unroll
        for (int yy = 0; yy < YY; ++yy)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              t[yy][mt][j] = y0 + yy < n_c
                                 ? __ldcg(mine0 + (size_t)(y0 + yy) * PER + mt * 128 + j * 32)
                                 : 0.f;
#pragma unroll
        for (int yy = 0; yy < YY; ++yy)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (y0 + yy < n_c) tot[mt][j] += t[yy][mt][j];
      }
      consumer_sync();   // every consumer has read the flag before it is reused
      if (threadIdx.x == 0) a.split_cnt[b] = 0u;
    }

    // ---------------------------------------------------- final epilogue of block b
    if (a.xscale.partial) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tok = token_of(mt, j);
          if (tok < a.M) tot[mt][j] *= s_r[tok];
        }
    }
    if constexpr (EPI == EPI_QKV) {
      const QkvOut& qo = a.qkv;
      const int D = qo.head_dim, half = D / 2;
      const int64_t pbase = qo.base_dev ? (int64_t)*qo.base_dev : qo.base;
      const size_t head_stride = (size_t)qo.page_size * D;
      const size_t page_stride = (size_t)qo.n_heads_kv * head_stride;
      const size_t layer_off = (size_t)qo.layer * qo.n_pages * page_stride;
      const int rlo = r0 + lo + pg, rhi = r0 + hi + pg;   // rows within the segment
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tok = token_of(mt, j);
          if (tok >= a.M || rlo >= seg_rows) continue;
          const float vlo = tot[mt][j], vhi = tot[mt][j + 2];
          const int64_t kvpos = pbase + qo.slot0 + tok;
          const size_t slot_off = layer_off +
                                  (size_t)qo.page_table[kvpos / qo.page_size] * page_stride +
                                  (size_t)(kvpos % qo.page_size) * D;
          if (seg < 2) {
            const int head = rlo / D, ii = rlo % D;   // ii < D / 2
            const int64_t pos = pbase + (qo.depth ? qo.depth[tok] : qo.slot0 + tok);
            const float2 cs = qo.rope[(pos < qo.max_pos ? pos : qo.max_pos - 1) * half + ii];
            const float y1 = vlo * cs.x - vhi * cs.y;
            const float y2 = vhi * cs.x + vlo * cs.y;
            uint16_t* dst = seg == 0 ? qo.q_out + ((size_t)tok * qo.n_heads_q + head) * D
                                     : qo.k_cache + slot_off + (size_t)head * head_stride;
            dst[ii] = f32_to_bf16_bits(y1);
            dst[ii + half] = f32_to_bf16_bits(y2);
          } else {
            qo.v_cache[slot_off + (size_t)(rlo / D) * head_stride + rlo % D] = f32_to_bf16_bits(vlo);
            if (rhi < seg_rows)
              qo.v_cache[slot_off + (size_t)(rhi / D) * head_stride + rhi % D] =
                  f32_to_bf16_bits(vhi);
          }
        }
    } else if constexpr (GLU) {
      // up tiles (warps 4..7) hand their sums to the gate tiles (warps 0..3)
      float* up = epi;   // [4 warps][MT][4][32]
      if (warp >= 4) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j) up[((warp - 4) * MT + mt) * 128 + j * 32 + lane] = tot[mt][j];
      }
      consumer_sync();
      if (warp < 4) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int tok = token_of(mt, j);
            const int row = r0 + ((j & 2) ? hi : lo) + pg;
            if (tok >= a.M || row >= a.N) continue;
            const float vu = up[(warp * MT + mt) * 128 + j * 32 + lane];
            reinterpret_cast<__nv_bfloat16*>(a.Y)[(int64_t)tok * a.ldy + row] =
                __float2bfloat16_rn(silu_f(tot[mt][j]) * vu);
          }
      }
      consumer_sync();   // the exchange buffer is free again
    } else {
      float ss[MT][2] = {};
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tok = token_of(mt, j);
          const int rs = r0 + ((j & 2) ? hi : lo) + pg;
          if (tok >= a.M || rs >= seg_rows) continue;
          const int row = seg_start + rs;
          const int64_t o = (int64_t)tok * a.ldy + row;
          const float v = tot[mt][j];
          if constexpr (EPI == EPI_BF16) {
            reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(v);
          } else if constexpr (EPI == EPI_F32) {
            reinterpret_cast<float*>(a.Y)[o] = v;
          } else {   // EPI_RESID
            const float xnew = yold[mt][j] + v;
            reinterpret_cast<float*>(a.Y)[o] = xnew;
            if (a.norm.xn) {
              a.norm.xn[o] = f32_to_bf16_bits(xnew * bf16_bits_to_f32(a.norm.gain[row]));
              ss[mt][j & 1] = fmaf(xnew, xnew, ss[mt][j & 1]);
            }
          }
        }
      if constexpr (EPI == EPI_RESID) {
        if (a.norm.xn && r0 + lo < seg_rows) {
          // sums of squares per token over this warp's 16-row tile, one part per tile
          float* const part = a.norm.partial + (size_t)((r0 + lo) / 16) * 16;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int jb = 0; jb < 2; ++jb) {
              float v = ss[mt][jb];
              v += __shfl_xor_sync(0xffffffffu, v, 4);
              v += __shfl_xor_sync(0xffffffffu, v, 8);
              v += __shfl_xor_sync(0xffffffffu, v, 16);
              if (g == 0) part[token_of(mt, jb)] = v;
            }
        }
      }
    }
  }
}

// ------------------------------------------------------------------- host --
namespace {
template <bool W4, int MT, int QB = 4>
cudaError_t tma_attr_all();
template <bool W4, int MT, int EPI, int QB>
cudaError_t tma_attr();
}  // namespace

// Shared-memory opt-in of every TMA GEMV instantiation and the tensor-map
// encoder lookup, once per process (before any stream capture: model creation
// calls this).
int32_t gemv_init() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const cudaError_t e[8] = {tma_attr_all<false, 1>(),   tma_attr_all<false, 2>(),
                              tma_attr_all<true, 1>(),    tma_attr_all<true, 2>(),
                              tma_attr_all<true, 1, 2>(), tma_attr_all<true, 2, 2>(),
                              tma_attr_all<true, 1, 3>(), tma_attr_all<true, 2, 3>()};
    // int4 codes, bf16 output, 17..32 activation rows
    const cudaError_t wide[1] = {tma_attr<true, 4, EPI_BF16, 4>()};
    for (cudaError_t x : e)
      if (x != cudaSuccess && err == cudaSuccess) err = x;
    for (cudaError_t x : wide)
      if (x != cudaSuccess && err == cudaSuccess) err = x;
  });
  if (err != cudaSuccess) return fail(SUB_ECUDA, std::string("gemv_init: ") + cudaGetErrorString(err));
  return SUB_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over a row-major [rows, cols] array with the given row stride.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, int64_t cols,
              int64_t rows, int64_t stride_bytes, int box_cols, int box_rows, int swz) {
  auto fn = encode_fn();
  if (!fn || !aligned16(ptr) || stride_bytes % 16 || (int64_t)box_cols * esize % 16) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)stride_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                       : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <bool W4, int MT, int EPI, int QB>
cudaError_t tma_attr() {
  return cudaFuncSetAttribute(gemv_tma_kernel<W4, MT, EPI, QB>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TmaGeom<W4, MT, QB>::SMEM);
}
template <bool W4, int MT, int QB>
cudaError_t tma_attr_all() {
  const cudaError_t e[5] = {tma_attr<W4, MT, EPI_BF16, QB>(), tma_attr<W4, MT, EPI_F32, QB>(),
                            tma_attr<W4, MT, EPI_RESID, QB>(), tma_attr<W4, MT, EPI_GLU, QB>(),
                            tma_attr<W4, MT, EPI_QKV, QB>()};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

template <bool W4, int MT, int EPI, int QB>
int32_t tma_launch(const GemvArgs& a, const TmaMaps& maps, const TmaPlan& pl, int grid,
                   cudaStream_t st) {
  SUB_TRY(gemv_init());
  SUB_CUDA_TRY(launch_k(gemv_tma_kernel<W4, MT, EPI, QB>, dim3(grid), dim3(W4 ? NTHR_W4 : NTHR),
                        TmaGeom<W4, MT, QB>::SMEM, st, maps, a, pl));
  return SUB_OK;
}

template <bool W4, int MT, int QB = 4>
int32_t tma_epi(const GemvArgs& a, int epi, const TmaMaps& maps, const TmaPlan& pl, int grid,
                cudaStream_t st) {
  switch (epi) {
    case EPI_BF16: return tma_launch<W4, MT, EPI_BF16, QB>(a, maps, pl, grid, st);
    case EPI_F32: return tma_launch<W4, MT, EPI_F32, QB>(a, maps, pl, grid, st);
    case EPI_RESID: return tma_launch<W4, MT, EPI_RESID, QB>(a, maps, pl, grid, st);
    case EPI_GLU: return tma_launch<W4, MT, EPI_GLU, QB>(a, maps, pl, grid, st);
    case EPI_QKV: return tma_launch<W4, MT, EPI_QKV, QB>(a, maps, pl, grid, st);
  }
  return fail(SUB_EINVAL, "bad gemv epilogue");
}

}  // namespace

static int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  });
  return n;
}

// Token tiles of 8 activation rows a launch uses: 1 or 2 up to 16 rows, then
// 4 (int4 codes, bf16 output) up to 32.  Six tiles (48 rows) leave room for
// only two stages and ran no faster than the tensor-core GEMM.
static int tma_tiles(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : 4; }

// Plan of a TMA launch, or false when the shape or the scratch does not fit
// (the caller then uses the register-streamed kernel).
static bool tma_plan(const GemvArgs& a, bool w4, int epi, TmaPlan* pl, int* grid) {
  const bool glu = epi == EPI_GLU;
  if (a.M < 1 || a.M > 32 || a.n_seg < 1 || a.n_seg > 3) return false;
  // past 16 rows: int4 codes with a bf16 output only (four token tiles)
  if (a.M > 16 && !(w4 && code_bits(a) == 4 && epi == EPI_BF16)) return false;
  if (glu && a.n_seg != 2) return false;
  const int G = (a.K + 63) / 64;
  if (w4 && G % 8) return false;   // scale/zero rows must be whole 16-byte strides
  if (a.K % 64) return false;      // X moves in whole 64-column slices
  if (epi == EPI_QKV && (BR % a.qkv.head_dim || a.qkv.head_dim < 16)) return false;
  if (epi == EPI_RESID && a.norm.xn && a.n_seg != 1) return false;   // tiles index one segment
  const int kc = w4 ? 512 : 128;
  pl->s_blk = (a.K + kc - 1) / kc;
  int nb = 0;
  for (int s = 0; s < 3; ++s) {
    if (s < (glu ? 1 : a.n_seg)) {
      const int rows = glu ? a.N : a.seg_end[s] - (s ? a.seg_end[s - 1] : 0);
      nb += (rows + (glu ? BR / 2 : BR) - 1) / (glu ? BR / 2 : BR);
    }
    pl->blk_end[s] = nb;
  }
  pl->n_blocks = nb;
  pl->n_maps = glu ? 2 : a.n_seg;
  pl->total = nb * pl->s_blk;
  *grid = std::min(pl->total, sm_count());
  // a CTA covers at least floor(total / grid) units, so a block of s_blk
  // units meets at most ceil(s_blk / that) + 1 CTAs
  pl->maxc = (pl->s_blk + pl->total / *grid - 1) / (pl->total / *grid) + 1;
  const int mt = tma_tiles(a.M);
  const size_t need = (size_t)nb * pl->maxc * NCW * mt * 128;
  return a.split_part && a.split_cnt && need <= a.split_cap && nb <= a.split_cnt_cap;
}

int32_t launch_gemv_tma(const GemvArgs& a, bool w4, int epi, cudaStream_t st, bool* done) {
  *done = false;
  static const bool on = env_flag("SUB_GEMV_TMA", true);
  if (!on) return SUB_OK;
  TmaPlan pl{};
  int grid = 0;
  if (!tma_plan(a, w4, epi, &pl, &grid)) return SUB_OK;
  const bool glu = epi == EPI_GLU;
  const int mt = tma_tiles(a.M);
  const int box_rows = glu ? BR / 2 : BR;
  const int G = (a.K + 63) / 64;
  const int bits = w4 ? code_bits(a) : 16;
  if (w4 && bits != 2 && bits != 3 && bits != 4) return SUB_OK;
  TmaMaps maps;
  memset(&maps, 0, sizeof(maps));
  for (int s = 0; s < (glu ? 2 : a.n_seg); ++s) {
    const int64_t rows = glu ? a.N : a.seg_end[s] - (s ? a.seg_end[s - 1] : 0);
    bool ok;
    if (w4) {
      // codes: G groups of 8 * bits bytes per row; 3-bit rows also get the
      // 64-byte box over the same bytes
      const int64_t cb = (int64_t)G * 8 * bits;
      ok = make_map(&maps.w[s], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.W[s], cb, rows, cb, 128,
                    box_rows, 128) &&
           (bits != 3 || make_map(&maps.w64[s], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.W[s], cb, rows,
                                  cb, 64, box_rows, 64)) &&
           make_map(&maps.s[s], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.S[s], G, rows,
                    (int64_t)G * 2, 8, box_rows, 0) &&
           make_map(&maps.z[s], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Z[s], G, rows,
                    (int64_t)G * 2, 8, box_rows, 0);
    } else {
      ok = make_map(&maps.w[s], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W[s], a.K, rows,
                    (int64_t)a.K * 2, 64, box_rows, 128);
    }
    if (!ok) return SUB_OK;
  }
  {
    // X [M, K] as [K/64][M][64]: a stage's 64-column slices land one after
    // another (the layout the consumers read), rows past M as zeros
    auto fn = encode_fn();
    if (!fn || !aligned16(a.X) || a.ldx % 8) return SUB_OK;
    const int xboxes = w4 ? 8 : 2;
    const cuuint64_t dims[3] = {64, (cuuint64_t)a.M, (cuuint64_t)(a.K / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)a.ldx * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)(mt * 8), (cuuint32_t)xboxes};
    const cuuint32_t es[3] = {1, 1, 1};
    if (fn(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.X), dims, strides,
           box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SUB_OK;
  }
  *done = true;
  if (w4 && bits == 2) return mt == 1 ? tma_epi<true, 1, 2>(a, epi, maps, pl, grid, st)
                                      : tma_epi<true, 2, 2>(a, epi, maps, pl, grid, st);
  if (w4 && bits == 3) return mt == 1 ? tma_epi<true, 1, 3>(a, epi, maps, pl, grid, st)
                                      : tma_epi<true, 2, 3>(a, epi, maps, pl, grid, st);
  if (w4 && mt > 2) return tma_launch<true, 4, EPI_BF16, 4>(a, maps, pl, grid, st);   // bf16 output only
  if (w4) return mt == 1 ? tma_epi<true, 1>(a, epi, maps, pl, grid, st)
                         : tma_epi<true, 2>(a, epi, maps, pl, grid, st);
  return mt == 1 ? tma_epi<false, 1>(a, epi, maps, pl, grid, st)
                 : tma_epi<false, 2>(a, epi, maps, pl, grid, st);
}

size_t gemv_tma_scratch_floats(const GemvArgs& a, bool w4, int epi) {
  GemvArgs t = a;
  t.split_part = reinterpret_cast<float*>(16);
  t.split_cnt = reinterpret_cast<unsigned int*>(16);
  t.split_cap = ~(size_t)0 >> 1;
  t.split_cnt_cap = 1 << 30;
  TmaPlan pl{};
  int grid = 0;
  if (!tma_plan(t, w4, epi, &pl, &grid)) return 0;
  return (size_t)pl.n_blocks * pl.maxc * NCW * tma_tiles(a.M) * 128;
}

// ------------------------------------------------------ bounded-wait check --
namespace {
__device__ unsigned int g_selftest_polls;   // polls the self-test wait made (0 = gave up)

// One thread waits, bounded, on an mbarrier that nothing arrives on and no
// copy is aimed at: the wait must give up after `limit` polls and the kernel
// must end normally.
__global__ void bounded_wait_selftest_kernel(uint32_t limit) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  g_selftest_polls = mbar_wait_polls(b, 0, limit);
}
}  // namespace

int32_t bounded_wait_selftest(uint32_t limit, uint32_t* polls) {
  SUB_CUDA_TRY(launch_k(bounded_wait_selftest_kernel, dim3(1), dim3(1), 0, nullptr, limit));
  SUB_CUDA_TRY(cudaStreamSynchronize(nullptr));
  SUB_CUDA_TRY(cudaMemcpyFromSymbol(polls, g_selftest_polls, sizeof(unsigned int)));
  return SUB_OK;
}

int32_t gemv_tma_timeouts(unsigned int* out) {
  SUB_CUDA_TRY(cudaMemcpyFromSymbol(out, g_tma_timeouts, sizeof(unsigned int)));
  return SUB_OK;
}

}  // namespace sub
