// Tree-shaped products (M > 16 activation rows: the verify pass over all tree
// nodes, the prompt prefill) on the 5th-generation tensor cores.
//
// Y[m, n] = sum_k X[m, k] W[n, k] with bf16 operands and fp32 accumulation,
// computed transposed (swap-AB): the MMA's A operand is a 128-row tile of W
// and its B operand a tile of up to 256 activation rows, so the accumulator
// D[n, m] sits in tensor memory with one weight row per TMEM lane and the
// tokens along the columns.  In the epilogue a warp reads 32 lanes (32
// consecutive weight rows) of a token column, so its global stores of Y[m, n]
// are coalesced.
//
// Persistent CTAs, one per SM at most, take the work items (token tile,
// weight tile, split of K) round-robin.  Warps 0..3 run the epilogue (one
// TMEM lane quarter each); the next warp's lane 0 streams K chunks of 64
// columns (128 bytes per row, the TMA 128-byte swizzle atom) of both operands
// into an S-stage shared-memory ring by TMA, and the last warp's lane 0 issues
// tcgen05.mma (kind::f16, M = 128, N = token tile, K = 16 per instruction)
// from the stages, handing each stage back with tcgen05.commit to its empty
// mbarrier.  The fp32 sums of consecutive items alternate between two TMEM
// accumulators (256 columns each): a commit marks one full, the epilogue
// reads it with tcgen05.ld and marks it empty, so the epilogue of one item
// overlaps the mainloop of the next and the ring never drains between items.
// Long K with few weight tiles splits over items; the last split of a tile
// adds the fp32 partials in split order.  Weight tiles never straddle a
// segment (q/k/v stacked, or gate/up for SiLU-GLU: 64 gate rows + 64 up rows
// per tile, the up half handed to the gate half through shared memory).
//
// Int4 weights (group 64, one group per K chunk): TMA moves the packed codes
// (32 bytes per row and chunk, 32-byte swizzle) beside the activations, and
// four converter warps (one thread per row) turn them into the bf16 A tile,
// bf16((q - z) * s) for their row's group scale and zero, written straight
// into the 128-byte swizzled layout the MMA descriptor reads.  Each converter
// fences its shared-memory writes into the async proxy and arrives on the
// stage's converted barrier, which the MMA lane waits on as well as the TMA
// barrier.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <mutex>
#include "gemm.cuh"

namespace sub {

namespace {

constexpr int TC_BM = 128;                 // weight rows per tile (TMEM lanes)
constexpr int TC_BK = 64;                  // K columns per stage (128 B per row)
constexpr int TC_TN = 256;                 // token rows per tile (max MMA N)
constexpr int A_BYTES = TC_BM * TC_BK * 2;     // 16 KB
constexpr int B_BYTES = TC_TN * TC_BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TC_STAGES = 4;
constexpr int XCH_BYTES = 64 * 64 * 4;     // GLU epilogue exchange: 64 up rows x 64 tokens
constexpr int TC_SMEM = 1024 + TC_STAGES * STAGE_BYTES + XCH_BYTES + 256;   // + barriers, TMEM address
constexpr int TMEM_COLS = 2 * TC_TN;       // two accumulators
// int4 weights: the stage also holds the packed codes of its 128 rows
constexpr int Q_BYTES = TC_BM * 32;                              // 4 KB
constexpr int STAGE_BYTES_W4 = A_BYTES + B_BYTES + Q_BYTES;      // 52 KB
constexpr int TC_EPI_WARPS = 4;                                  // one per TMEM lane quarter
constexpr int TC_CONV_WARPS = 4;                                 // one thread per row
constexpr int TC_THREADS = (TC_EPI_WARPS + 2) * 32;              // + producer, MMA issuer
constexpr int TC_THREADS_W4 = (TC_EPI_WARPS + TC_CONV_WARPS + 2) * 32;
constexpr int TC_SMEM_W4 = 1024 + TC_STAGES * STAGE_BYTES_W4 + XCH_BYTES + 256;
static_assert(8 * (3 * TC_STAGES + 4) + 4 <= 256, "barriers and the TMEM address fit the tail");
static_assert(STAGE_BYTES_W4 % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(TC_SMEM_W4 <= 227 * 1024, "int4 ring must fit one CTA's shared memory");

__device__ unsigned int g_tc_timeouts;   // waits that ran out (never expected)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: a wait that runs out records itself and returns (wrong
// numbers and a host-visible count rather than a hang).
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 22); ++i)
    if (mbar_try_wait(bar, parity)) return;
  atomicAdd(&g_tc_timeouts, 1u);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05 --
// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout TMA writes (8-row groups of 1024 bytes): start address,
// leading byte offset (unused by swizzled K-major: 16), stride byte offset
// 1024 between 8-row groups, the descriptor version bit, swizzle mode 2.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// The four epilogue warps (0..3) meet here; other warps may still be running.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// One word of eight 4-bit codes (byte p: element 2p in the low nibble, 2p+1
// in the high one) to eight bf16 weights (q - z) * s, each rounded once to
// fp32 by the subtraction (exact) and the product, then to bf16.
__device__ __forceinline__ uint4 dequant8(uint32_t w, float s, float z) {
  uint32_t out[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    // 2^23 + q as an fp32 bit pattern, minus 2^23: the code as an exact float
    const float q0 = __uint_as_float(0x4B000000u | ((w >> (8 * p)) & 15u)) - 8388608.0f;
    const float q1 = __uint_as_float(0x4B000000u | ((w >> (8 * p + 4)) & 15u)) - 8388608.0f;
    const float d0 = __fmul_rn(__fsub_rn(q0, z), s);
    const float d1 = __fmul_rn(__fsub_rn(q1, z), s);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out[p]) : "f"(d1), "f"(d0));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(TC_BM >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 16 consecutive columns of fp32 from TMEM, one lane per thread.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace

struct TcMaps {   // aligned as its CUtensorMap members
  CUtensorMap w[3];   // weight segments: [rows, K] bf16, box 64 x (128 or 64 rows);
                      // int4: packed codes [rows, K/2] bytes, box 32 x (128 or 64 rows)
  CUtensorMap x;      // activations [M, K] bf16, box 64 x token-tile rows
};

struct TcPlan {
  int blk_end[3];     // cumulative weight tiles per segment
  int n_maps;
  int chunks;         // K chunks of 64 columns
  int per_split;      // chunks per split of K
  int xrows;          // token rows of the activation box
  int ntx, nty, ks;   // token tiles, weight tiles, splits of K
  int items;          // ntx * nty * ks work items, shared round-robin by the CTAs
};

template <int EPI, bool W4>
__global__ void __launch_bounds__(W4 ? TC_THREADS_W4 : TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, const GemvArgs a, const TcPlan pl) {
  constexpr bool GLU = EPI == EPI_GLU;
  constexpr int HALF = GLU ? TC_BM / 2 : TC_BM;   // rows of one segment in a tile
  constexpr int SB = W4 ? STAGE_BYTES_W4 : STAGE_BYTES;
  constexpr int PROD_WARP = TC_EPI_WARPS + (W4 ? TC_CONV_WARPS : 0);
  constexpr int MMA_WARP = PROD_WARP + 1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  float* const xch = reinterpret_cast<float*>(base_ptr + TC_STAGES * SB);   // GLU exchange
  // full[S], empty[S], converted[S], accumulator full[2], accumulator empty[2]
  const uint32_t bars = base + TC_STAGES * SB + XCH_BYTES;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (TC_STAGES + s); };
  auto conv_bar = [&](int s) { return bars + 8u * (2 * TC_STAGES + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (3 * TC_STAGES + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (3 * TC_STAGES + 2 + b); };
  uint32_t* const tmem_slot =
      reinterpret_cast<uint32_t*>(base_ptr + TC_STAGES * SB + XCH_BYTES + 8 * (3 * TC_STAGES + 4));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item w -> token tile, weight tile, split of K (token tiles fastest,
  // so the CTAs running one weight tile's token tiles share it in L2)
  struct Item {
    int tok0, tn, tile, seg, r0, kz, c0, nck;
  };
  auto item = [&](int w) {
    Item d;
    const int tx = w % pl.ntx, rest = w / pl.ntx;
    d.tile = rest % pl.nty;
    d.kz = rest / pl.nty;
    d.tok0 = tx * TC_TN;
    d.tn = min(TC_TN, ((a.M - d.tok0) + 15) / 16 * 16);   // MMA N (multiple of 16)
    d.seg = 0;
    while (d.seg < 2 && d.tile >= pl.blk_end[d.seg]) ++d.seg;
    d.r0 = (d.tile - (d.seg ? pl.blk_end[d.seg - 1] : 0)) * HALF;   // first row in the segment
    d.c0 = d.kz * pl.per_split;
    d.nck = max(0, min(pl.chunks, d.c0 + pl.per_split) - d.c0);
    return d;
  };
  const int ks = pl.ks;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(conv_bar(s), TC_CONV_WARPS * 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), TC_EPI_WARPS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The producer and the MMA issuer are lane 0 of their warps; the other
  // lanes go straight to the final barrier, so they never compete with the
  // working lane's instruction stream.
  if (warp == PROD_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      auto issue = [&](const Item& d, int i, int it, bool weights, bool acts) {
        const int s = it % TC_STAGES, c = d.c0 + i, kx = c * TC_BK;
        const uint32_t st = base + s * SB, fb = full_bar(s);
        if (weights) {
          mbar_expect_tx(fb, W4 ? Q_BYTES + B_BYTES : STAGE_BYTES);
          for (int h = 0; h < (GLU ? 2 : 1); ++h) {
            if constexpr (W4)
              tma_load_2d(st + A_BYTES + B_BYTES + h * HALF * 32, &maps.w[GLU ? h : d.seg], c * 32,
                          d.r0, fb);
            else
              tma_load_2d(st + h * HALF * 128, &maps.w[GLU ? h : d.seg], kx, d.r0, fb);
          }
        }
        if (acts) {
          // the activation box always moves TC_TN rows' worth of bytes: rows past
          // the tensor (and past the box) arrive as zeros
          for (int y = 0; y < TC_TN; y += pl.xrows)
            tma_load_2d(st + A_BYTES + y * 128, &maps.x, kx, d.tok0 + y, fb);
        }
      };
      int it = 0;   // chunks issued so far (stage it % S, round it / S)
      int w = blockIdx.x;
      if (w < pl.items) {
        // the first item's first stages: weights before the wait on the
        // producing kernel, activations after it
        const Item d = item(w);
        const int npre = min(TC_STAGES, d.nck);
        for (int i = 0; i < npre; ++i) issue(d, i, i, true, false);
        pdl_wait();
        for (int i = 0; i < npre; ++i) issue(d, i, i, false, true);
        it = npre;
        for (int i = npre; i < d.nck; ++i, ++it) {
          mbar_wait(empty_bar(it % TC_STAGES), ((it / TC_STAGES) - 1) & 1);
          issue(d, i, it, true, true);
        }
        for (w += gridDim.x; w < pl.items; w += gridDim.x) {
          const Item e = item(w);
          for (int i = 0; i < e.nck; ++i, ++it) {
            if (it >= TC_STAGES) mbar_wait(empty_bar(it % TC_STAGES), ((it / TC_STAGES) - 1) & 1);
            issue(e, i, it, true, true);
          }
        }
      } else {
        pdl_wait();
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      int it = 0, t = 0;   // chunks consumed, items done
      for (int w = blockIdx.x; w < pl.items; w += gridDim.x, ++t) {
        const Item d = item(w);
        const int ab = t & 1;
        // accumulator ab is free once the epilogue has read item t - 2
        if (t >= 2) mbar_wait(acce_bar(ab), ((t >> 1) - 1) & 1);
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(ab * TC_TN);
        const uint32_t idesc = idesc_bf16(d.tn);
        for (int i = 0; i < d.nck; ++i, ++it) {
          const int s = it % TC_STAGES;
          mbar_wait(full_bar(s), (it / TC_STAGES) & 1);
          if constexpr (W4) mbar_wait(conv_bar(s), (it / TC_STAGES) & 1);
          tc_fence_after();
          const uint32_t st = base + s * SB;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            tc_mma(acc, smem_desc_sw128(st + kk * 32), smem_desc_sw128(st + A_BYTES + kk * 32),
                   idesc, (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit(empty_bar(s));   // the stage is free once these MMAs have read it
        }
        tc_commit(accf_bar(ab));     // the item's sums are complete
      }
    }
  } else if (W4 && warp >= TC_EPI_WARPS) {
    // ---------------------------------------------------------- converters
    // thread = row of the tile; the group's scale and zero come one chunk ahead
    const int rr = threadIdx.x - TC_EPI_WARPS * 32;
    const int G = (a.K + TC_BK - 1) / TC_BK;   // groups per row = K chunks
    int it = 0;
    for (int w = blockIdx.x; w < pl.items; w += gridDim.x) {
      const Item d = item(w);
      const int sseg = GLU ? (rr >= HALF ? 1 : 0) : d.seg;
      const int rs = d.r0 + (GLU ? (rr & (HALF - 1)) : rr);
      const int rows = GLU ? a.N : a.seg_end[sseg] - (sseg ? a.seg_end[sseg - 1] : 0);
      const bool ok = rs < rows;
      const uint16_t* const sp = a.S[sseg] + (int64_t)(ok ? rs : 0) * G;
      const uint16_t* const zp = a.Z[sseg] + (int64_t)(ok ? rs : 0) * G;
      uint16_t sv = 0, zv = 0;
      if (ok && d.nck > 0) {
        sv = __ldg(sp + d.c0);
        zv = __ldg(zp + d.c0);
      }
      for (int i = 0; i < d.nck; ++i, ++it) {
        const int s = it % TC_STAGES;
        const float sc = bf16_bits_to_f32(sv), zc = bf16_bits_to_f32(zv);
        if (ok && i + 1 < d.nck) {
          sv = __ldg(sp + d.c0 + i + 1);
          zv = __ldg(zp + d.c0 + i + 1);
        }
        mbar_wait(full_bar(s), (it / TC_STAGES) & 1);
        uint8_t* const st = base_ptr + s * SB;
        // the codes arrive with the 32-byte swizzle: 16-byte half h of row rr
        // sits at half h ^ ((rr >> 2) & 1), so eight consecutive rows of one
        // read phase cover all 32 banks
        const uint8_t* const qrow = st + A_BYTES + B_BYTES + rr * 32;
        const int flip = (rr >> 2) & 1;
        const uint4 q0 = *reinterpret_cast<const uint4*>(qrow + (flip << 4));
        const uint4 q1 = *reinterpret_cast<const uint4*>(qrow + ((1 ^ flip) << 4));
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint8_t* const arow = st + rr * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)   // 16-byte chunk c of the row sits at chunk c ^ (row % 8)
          *reinterpret_cast<uint4*>(arow + ((c ^ (rr & 7)) << 4)) = dequant8(words[c], sc, zc);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(conv_bar(s));
      }
    }
  } else if (warp < TC_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    pdl_wait();   // the epilogue reads what earlier kernels wrote
    const int lrow = warp * 32 + lane;   // TMEM lane = row of the tile
    int t = 0;
    for (int w = blockIdx.x; w < pl.items; w += gridDim.x, ++t) {
      const Item d = item(w);
      const int ab = t & 1;
      mbar_wait(accf_bar(ab), (t >> 1) & 1);
      // Dependents may launch once this CTA's last mainloop is done.  Only
      // threads past their own wait signal it: a later kernel reads some
      // inputs before its wait (the tree of the attention kernel) and counts on
      // everything before this kernel's predecessor having finished; and
      // dependents launched earlier would sit on these SMs for the whole
      // persistent run.
      if (w + (int)gridDim.x >= pl.items) pdl_trigger();
      __syncwarp();
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)(ab * TC_TN) + ((uint32_t)(warp * 32) << 16);
      const int seg = d.seg, r0 = d.r0, tok0 = d.tok0, tn = d.tn, nck = d.nck, kz = d.kz;
      const int seg_rows = GLU ? a.N : a.seg_end[seg] - (seg ? a.seg_end[seg - 1] : 0);
      const int seg_start = GLU ? 0 : (seg ? a.seg_end[seg - 1] : 0);
      const int rs = r0 + (GLU ? (lrow & (HALF - 1)) : lrow);     // row within the segment
      const bool row_ok = rs < seg_rows;
      const int n_glob = seg_start + rs;

      // split of K: park fp32 partials [tile][split][token][row], the last split sums
      bool last = true;
      float* part = nullptr;
      if (ks > 1) {
        const size_t tile_lin = (size_t)d.tile * pl.ntx + (size_t)(tok0 / TC_TN);
        part = a.split_part + tile_lin * ks * (size_t)(TC_TN * TC_BM);
        float* mine = part + (size_t)kz * (TC_TN * TC_BM);
        for (int cb = 0; cb < tn; cb += 16) {
          float v[16];
          if (nck > 0) tc_ld16(taddr + cb, v);
          else
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(mine + (size_t)(cb + j) * TC_BM + lrow, v[j]);
        }
        __shared__ unsigned int s_last;
        epi_bar();
        if (threadIdx.x == 0) {
          __threadfence();
          s_last = (atomicAdd(a.split_cnt + tile_lin, 1u) == (unsigned)ks - 1) ? 1u : 0u;
          __threadfence();
        }
        epi_bar();
        last = s_last != 0;
        if (last && threadIdx.x == 0) a.split_cnt[tile_lin] = 0u;
      }

      if (last) {
        // 64 columns (tokens) per round: four TMEM loads, or four splits' worth of
        // partial sums, and all their global loads in flight together
        for (int cg = 0; cg < tn; cg += 64) {
          const int ncol = min(64, tn - cg);   // a multiple of 16
          float v[64];
          if (ks > 1) {
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = 0.f;
            for (int z = 0; z < ks; ++z) {
              float p[64];
#pragma unroll
              for (int j = 0; j < 64; ++j)
                p[j] = j < ncol ? __ldcg(part + ((size_t)z * TC_TN + cg + j) * TC_BM + lrow) : 0.f;
#pragma unroll
              for (int j = 0; j < 64; ++j) v[j] += p[j];
            }
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float tv[16];
              if (q * 16 < ncol && nck > 0) tc_ld16(taddr + cg + q * 16, tv);
              else
#pragma unroll
                for (int j = 0; j < 16; ++j) tv[j] = 0.f;
#pragma unroll
              for (int j = 0; j < 16; ++j) v[q * 16 + j] = tv[j];
            }
          }
          if constexpr (GLU) {
            // up rows (lanes 64..127) hand their values to the gate rows (lanes 0..63)
            epi_bar();
            if (lrow >= HALF)
#pragma unroll
              for (int j = 0; j < 64; ++j) xch[j * HALF + (lrow - HALF)] = v[j];
            epi_bar();
            if (lrow < HALF && row_ok) {
#pragma unroll
              for (int j = 0; j < 64; ++j) {
                const int m = tok0 + cg + j;
                if (j < ncol && m < a.M)
                  reinterpret_cast<__nv_bfloat16*>(a.Y)[(int64_t)m * a.ldy + rs] =
                      __float2bfloat16_rn(silu_f(v[j]) * xch[j * HALF + lrow]);
              }
            }
          } else if (row_ok) {
            if constexpr (EPI == EPI_RESID) {
              // all old values first: a load after a store to Y would wait for it
              float* const Y = reinterpret_cast<float*>(a.Y);
              float y[64];
#pragma unroll
              for (int j = 0; j < 64; ++j) {
                const int m = tok0 + cg + j;
                y[j] = (j < ncol && m < a.M) ? __ldcg(Y + (int64_t)m * a.ldy + n_glob) : 0.f;
              }
#pragma unroll
              for (int j = 0; j < 64; ++j) {
                const int m = tok0 + cg + j;
                if (j < ncol && m < a.M) Y[(int64_t)m * a.ldy + n_glob] = y[j] + v[j];
              }
            } else {
#pragma unroll
              for (int j = 0; j < 64; ++j) {
                const int m = tok0 + cg + j;
                if (j >= ncol || m >= a.M) continue;
                const int64_t o = (int64_t)m * a.ldy + n_glob;
                if constexpr (EPI == EPI_BF16) {
                  reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(v[j]);
                } else {
                  reinterpret_cast<float*>(a.Y)[o] = v[j];
                }
              }
            }
          }
        }
      }
      // this item's accumulator may take item t + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(ab));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
}

// ------------------------------------------------------------------- host --
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
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

// 2-D bf16 map over a row-major [rows, cols] array, 64-column (128-byte) boxes
// with the 128-byte swizzle.
bool tc_map(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows, int64_t stride_bytes,
            int box_rows) {
  auto fn = tc_encode_fn();
  if (!fn || !aligned16(ptr) || stride_bytes % 16 || box_rows < 1 || box_rows > 256) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)stride_bytes};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte map over packed int4 codes [rows, row_bytes]: 32-byte boxes (one group of
// 64 codes per row), 32-byte swizzle.
bool tc_map_q(CUtensorMap* m, const void* ptr, int64_t row_bytes, int64_t rows, int box_rows) {
  auto fn = tc_encode_fn();
  if (!fn || !aligned16(ptr) || row_bytes % 32 || box_rows < 1 || box_rows > 256) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_sm_count() {
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

template <int EPI, bool W4>
int32_t tc_launch(const GemvArgs& a, const TcMaps& maps, const TcPlan& pl, dim3 grid,
                  cudaStream_t st) {
  SUB_TRY(gemm_tc_init());
  SUB_CUDA_TRY(launch_k(gemm_tc_kernel<EPI, W4>, grid, dim3(W4 ? TC_THREADS_W4 : TC_THREADS),
                        W4 ? TC_SMEM_W4 : TC_SMEM, st, maps, a, pl));
  return SUB_OK;
}

template <bool W4>
int32_t tc_dispatch(const GemvArgs& a, int epi, const TcMaps& maps, const TcPlan& pl, dim3 grid,
                    cudaStream_t st) {
  switch (epi) {
    case EPI_BF16: return tc_launch<EPI_BF16, W4>(a, maps, pl, grid, st);
    case EPI_F32: return tc_launch<EPI_F32, W4>(a, maps, pl, grid, st);
    case EPI_RESID: return tc_launch<EPI_RESID, W4>(a, maps, pl, grid, st);
    case EPI_GLU: return tc_launch<EPI_GLU, W4>(a, maps, pl, grid, st);
  }
  return fail(SUB_EINVAL, "bad gemm epilogue");
}

}  // namespace

int32_t gemm_tc_init() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const void* ks[8] = {
        (const void*)gemm_tc_kernel<EPI_BF16, false>, (const void*)gemm_tc_kernel<EPI_F32, false>,
        (const void*)gemm_tc_kernel<EPI_RESID, false>, (const void*)gemm_tc_kernel<EPI_GLU, false>,
        (const void*)gemm_tc_kernel<EPI_BF16, true>,  (const void*)gemm_tc_kernel<EPI_F32, true>,
        (const void*)gemm_tc_kernel<EPI_RESID, true>, (const void*)gemm_tc_kernel<EPI_GLU, true>};
    for (int i = 0; i < 8; ++i)
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   i < 4 ? TC_SMEM : TC_SMEM_W4);
  });
  if (err != cudaSuccess) return fail(SUB_ECUDA, std::string("gemm_tc_init: ") + cudaGetErrorString(err));
  return SUB_OK;
}

// Tile plan: weight tiles per segment, token tiles, splits of K.  False when
// the product is not for this kernel (the q/k/v epilogue, fused-norm outputs,
// a segment count or alignment it does not handle).
static bool tc_plan(const GemvArgs& a, bool w4, int epi, TcPlan* pl, dim3* grid, size_t* scratch) {
  static const bool on = env_flag("SUB_GEMM_TC", true);
  static const bool on_w4 = env_flag("SUB_GEMM_TC_W4", true);
  if (!on || (w4 && !on_w4) || epi == EPI_QKV || a.M <= 16 || a.xscale.partial) return false;
  if (epi == EPI_RESID && a.norm.xn) return false;
  const bool glu = epi == EPI_GLU;
  if (a.n_seg < 1 || a.n_seg > 3 || (glu && a.n_seg != 2)) return false;
  if (a.K % 8 || a.ldx % 8) return false;
  const int half = glu ? TC_BM / 2 : TC_BM;
  int nb = 0;
  for (int s = 0; s < 3; ++s) {
    if (s < (glu ? 1 : a.n_seg)) {
      const int rows = glu ? a.N : a.seg_end[s] - (s ? a.seg_end[s - 1] : 0);
      nb += (rows + half - 1) / half;
    }
    pl->blk_end[s] = nb;
  }
  pl->n_maps = glu ? 2 : a.n_seg;
  pl->chunks = (a.K + TC_BK - 1) / TC_BK;
  // activation box height: a power of two from 16 to TC_TN, so whole boxes
  // tile the TC_TN rows of a stage exactly
  pl->xrows = 16;
  while (pl->xrows < TC_TN && pl->xrows < a.M) pl->xrows *= 2;
  const int tok_tiles = (a.M + TC_TN - 1) / TC_TN;
  // split K while the splits still fit one wave of one CTA per SM (a round of
  // fp32 partials is cheaper than idle SMs), at least 16 chunks per split
  const int ctas = nb * tok_tiles;
  int ks = std::max(1, std::min(tc_sm_count() / ctas, std::min(8, pl->chunks / 16)));
  size_t need = ks > 1 ? (size_t)ctas * ks * TC_TN * TC_BM : 0;
  while (ks > 1 && (need > a.split_cap || ctas > a.split_cnt_cap || !a.split_part || !a.split_cnt)) {
    --ks;
    need = ks > 1 ? (size_t)ctas * ks * TC_TN * TC_BM : 0;
  }
  pl->per_split = (pl->chunks + ks - 1) / ks;
  ks = (pl->chunks + pl->per_split - 1) / pl->per_split;
  need = ks > 1 ? (size_t)ctas * ks * TC_TN * TC_BM : 0;
  pl->ntx = tok_tiles;
  pl->nty = nb;
  pl->ks = ks;
  pl->items = ctas * ks;
  *grid = dim3(std::min(pl->items, tc_sm_count()));   // persistent: one CTA per SM at most
  *scratch = need;
  return true;
}

size_t gemm_tc_scratch_floats(const GemvArgs& a, bool w4, int epi) {
  GemvArgs t = a;
  t.split_part = reinterpret_cast<float*>(16);
  t.split_cnt = reinterpret_cast<unsigned int*>(16);
  t.split_cap = ~(size_t)0 >> 1;
  t.split_cnt_cap = 1 << 30;
  TcPlan pl{};
  dim3 grid;
  size_t need = 0;
  return tc_plan(t, w4, epi, &pl, &grid, &need) ? need : 0;
}

int32_t launch_gemm_tc(const GemvArgs& a, bool w4, int epi, cudaStream_t st, bool* done) {
  *done = false;
  TcPlan pl{};
  dim3 grid;
  size_t need = 0;
  if (!tc_plan(a, w4, epi, &pl, &grid, &need)) return SUB_OK;
  const bool glu = epi == EPI_GLU;
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  for (int s = 0; s < pl.n_maps; ++s) {
    const int64_t rows = glu ? a.N : a.seg_end[s] - (s ? a.seg_end[s - 1] : 0);
    const int box = glu ? TC_BM / 2 : TC_BM;
    // int4 rows hold ceil(K/64) groups of 32 bytes (codes past K are 0 and meet
    // zero activations: the activation map ends at K)
    if (w4 ? !tc_map_q(&maps.w[s], a.W[s], (int64_t)pl.chunks * 32, rows, box)
           : !tc_map(&maps.w[s], a.W[s], a.K, rows, (int64_t)a.K * 2, box))
      return SUB_OK;
  }
  if (!tc_map(&maps.x, a.X, a.K, a.M, (int64_t)a.ldx * 2, pl.xrows)) return SUB_OK;
  *done = true;
  return w4 ? tc_dispatch<true>(a, epi, maps, pl, grid, st)
            : tc_dispatch<false>(a, epi, maps, pl, grid, st);
}

int32_t gemm_tc_timeouts(unsigned int* out) {
  SUB_CUDA_TRY(cudaMemcpyFromSymbol(out, g_tc_timeouts, sizeof(unsigned int)));
  return SUB_OK;
}

}  // namespace sub
