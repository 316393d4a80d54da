// Warp-level GEMV for draft-shaped products (M <= 16 rows of activations).
//
// Y[m, n] = sum_k X[m, k] W[n, k].  Swap-AB on mma.sync m16n8k16: a 16-row
// tile of W is the A operand and up to 8 activation rows are the B operand, so
// every weight byte is read exactly once, at full 128-bit (bf16) or 64-bit
// (int4) width, straight from HBM into registers.  The order of the K index
// inside one mma is free as long as A and B agree, so each lane loads its own
// contiguous run of K and the B fragment is built from the same run.  Each
// warp keeps U steps of weights in flight (a rolling register prefetch), and
// the first U steps are requested before the kernel waits on its predecessor
// (programmatic dependent launch), so weight streaming overlaps the previous
// kernel's tail.
//
// Int4 tiles compute, per 64-group, P = X . (128 + q) with q turned into the
// bf16 value 128+q by one bit-or (0x4300 | q), the group sum Sx = X . 1 by one
// more mma with an all-ones A, and fold the zero point and the scale in fp32:
// Y += s * (P - (128 + z) * Sx).  This is (q - z) * s without rounding the
// dequantised weight to bf16 first.
//
// A CTA owns RT row tiles (16 rows each) over one split of K (grid.y), with
// its slice of the activations staged once in shared memory; its 4 warps
// split the slice and their partial sums meet in shared memory in a fixed
// order, as do the splits, so results are deterministic.  Epilogues: bf16 or
// fp32 store, fp32 residual add (which can also produce the next RMSNorm's
// input in factored form, see NormOut), SiLU(gate)*up, and the q/k/v epilogue
// (RoPE on q and k from rows paired i / i + d/2 inside one tile, bf16 q out,
// k and v written into the paged KV cache).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include "common.cuh"

namespace sub {

enum GemvEpi : int {
  EPI_BF16 = 0,    // Y bf16 [M, ldy]
  EPI_F32 = 1,     // Y fp32 [M, ldy]
  EPI_RESID = 2,   // Y fp32 [M, ldy] += acc (optionally + next RMSNorm, see NormOut)
  EPI_GLU = 3,     // Y bf16 [M, ldy] = silu(gate) * up; segments 0 (gate) and 1 (up)
  EPI_QKV = 4,     // segments q, k, v -> RoPE, bf16 q, K/V into the cache (QkvOut)
};

// Residual epilogue extension (the next RMSNorm, factored): every unit writes
// xn[m, rows] = bf16(Y[m, rows] * gain[rows]) for its own rows and, for each
// 16-row tile t of the output, partial[t * 16 + m] = sum over the tile's rows
// of Y[m, row]^2.  The consumer GEMV forms the row scale itself (RowScale):
// RMSNorm is a per-row scalar, so sum_k W[n,k] x[m,k] r[m] g[k] =
// r[m] sum_k W[n,k] (x[m,k] g[k]), with the bf16 rounding taken before the scale.
// No grid-wide step is left in the producer: the consumer starts after it ends.
struct NormOut {
  uint16_t* xn;              // [M, ldy] bf16, or null for a plain residual add
  const uint16_t* gain;      // [ldy]
  float* partial;            // [ceil(ldy / 16) * 16] per-tile sums of squares
};

// Row scales of a factored RMSNorm, formed by the consumer from the producer's
// per-tile sums of squares: r[m] = rsqrt(sum_p partial[p * 16 + tok0 + m] /
// hidden + eps), the parts summed in one fixed order (row_scale below).
struct RowScale {
  const float* partial;      // null: no scale
  int n_parts;
  int hidden;
  float eps;
  int tok0;                  // token offset of the consumer's row 0
};

// r[m] for one token, computed by a whole warp (every lane returns it): lane l
// adds parts l, l + 32, ... in order, eight loads in flight per round, then a
// butterfly sum.  Every kernel that applies a RowScale uses this routine, so
// all of them see the same r.
__device__ inline float row_scale(const RowScale& rs, int m, int lane) {
  float t = 0.f;
  const float* p = rs.partial + rs.tok0 + m;
  for (int p0 = 0; p0 < rs.n_parts; p0 += 256) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int q = p0 + k * 32 + lane;
      v[k] = q < rs.n_parts ? __ldcg(p + (size_t)q * 16) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) t += v[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return rsqrtf(t / (float)rs.hidden + rs.eps);
}

// q/k/v epilogue: rows are q (Hq*D), k (Hkv*D), v (Hkv*D); token m sits at
// position base + depth[m] and its K/V go to cache position base + slot0 + m.
struct QkvOut {
  int n_heads_q, n_heads_kv, head_dim;
  const float2* rope;        // [max_pos, D/2] (cos, sin)
  int max_pos;
  const int32_t* depth;      // [M] or null (chain: slot0 + m)
  int slot0;
  int64_t base;
  const int32_t* base_dev;   // overrides base when non-null
  uint16_t* q_out;           // [M, Hq, D]
  uint16_t* k_cache;
  uint16_t* v_cache;
  const int32_t* page_table;
  int page_size, n_pages, layer;
};

struct GemvArgs {
  const uint16_t* X;     // [M, K] bf16, row stride ldx elements
  int M, K, ldx;
  // up to 4 weight segments stacked along N (rows); seg_end is cumulative
  const void* W[4];      // bf16 [rows, K]  or  packed int4 [rows, G*32]
  const uint16_t* S[4];  // int4 scales [rows, G]
  const uint16_t* Z[4];  // int4 zeros  [rows, G]
  int seg_end[4];
  int n_seg;
  int N;                 // rows covered by the grid (for GLU: rows of one segment)
  void* Y;               // output (bf16 or fp32)
  int ldy;
  RowScale xscale;       // per-row scale of the result (a factored RMSNorm), or none
  NormOut norm;          // EPI_RESID only
  QkvOut qkv;            // EPI_QKV only
  // split of K over CTAs (grid.y): partial sums meet in split_part and the
  // last CTA of a row unit adds them in split order; counters start at zero
  // and are left at zero.  split_cap = floats available in split_part.
  float* split_part;
  unsigned int* split_cnt;
  size_t split_cap;
  int split_cnt_cap;
  int ksplit;            // set by launch_gemv
  int bits;              // quantised weights: code bits 2, 3 or 4 (0 means 4)
};

// Codes of 2- and 3-bit substitutes spread into the int4 word layout (code i
// of a lane's run of 8 at bits 4i .. 4i+3), so one unpack serves all widths.
// spread2: eight 2-bit fields at stride 2 -> stride 4 (bit interleave by
// shift-or-mask); spread1: eight bits at stride 1 -> stride 4.
__device__ __forceinline__ uint32_t spread2(uint32_t v) {
  v &= 0xffffu;
  v = (v | (v << 8)) & 0x00ff00ffu;
  v = (v | (v << 4)) & 0x0f0f0f0fu;
  return (v | (v << 2)) & 0x33333333u;
}
__device__ __forceinline__ uint32_t spread1(uint32_t v) {
  v &= 0xffu;
  v = (v | (v << 12)) & 0x000f000fu;
  v = (v | (v << 6)) & 0x03030303u;
  return (v | (v << 3)) & 0x11111111u;
}

// Code bits of a quantised product (0 in GemvArgs means 4).
inline int code_bits(const GemvArgs& a) { return a.bits ? a.bits : 4; }

// Launch: quantised (is_w4; a.bits code bits) or bf16 weights, epilogue, M <= 16.
// Quantised codes of every width and bf16 weights take the TMA variant when
// it fits, else the register-streamed kernel.
int32_t launch_gemv(const GemvArgs& a, bool is_w4, int epi, cudaStream_t stream);
// Row units (CTAs along grid.x) a launch uses; NormOut::partial holds 16 floats per unit.
int gemv_grid(const GemvArgs& a, int epi);
// Splits of K over CTAs the launch would use given room for them (1 = no split).
int gemv_ksplit(const GemvArgs& a, bool is_w4, int epi);

// TMA-streamed variant (gemv_tma.cu): one producer warp fills a shared-memory
// ring by TMA, eight consumer warps (one 16-row tile each) multiply from it,
// one CTA per SM with the (block, K-stage) units split evenly.  Launches and
// sets *done when the shape and the split scratch allow it; otherwise leaves
// *done false and launches nothing.  launch_gemv tries it first
// (SUB_GEMV_TMA=0 turns it off).  Quantised codes (is_w4) are code_bits(a) wide.
int32_t launch_gemv_tma(const GemvArgs& a, bool is_w4, int epi, cudaStream_t stream, bool* done);
// Partial-sum floats the TMA variant needs in split_part (0: it would not run).
size_t gemv_tma_scratch_floats(const GemvArgs& a, bool is_w4, int epi);
// Kernel attributes of the TMA variant; call before any stream capture.
int32_t gemv_init();
// Pipeline waits that ran out since load (each one is a bug; never expected).
int32_t gemv_tma_timeouts(unsigned int* out);
// The CUDA driver API's tensor-map encoder (null if unavailable), and a 2-D tiled map
// over a row-major [rows, cols] array with the given row stride and box
// (swz: 0 for no swizzle, 64 or 128 for that swizzle span in bytes); false
// when the encoder or the alignment refuses.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, int64_t cols,
              int64_t rows, int64_t stride_bytes, int box_cols, int box_rows, int swz);
// One bounded wait on an mbarrier nothing arrives on; *polls = polls made
// before it was satisfied, 0 when it gave up after `limit` polls.
int32_t bounded_wait_selftest(uint32_t limit, uint32_t* polls);

}  // namespace sub
