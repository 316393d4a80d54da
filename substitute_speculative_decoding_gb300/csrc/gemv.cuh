// Warp-level GEMV for draft-shaped products (M <= 16 rows of activations).
//
// Y[m, n] = sum_k X[m, k] W[n, k].  Swap-AB on mma.sync m16n8k16: a 16-row
// tile of W is the A operand and up to 8 activation rows are the B operand, so
// every weight byte is read exactly once, at full 128-bit (bf16) or 64-bit
// (int4) width, straight from HBM into registers.  The order of the K index
// inside one mma is free as long as A and B agree, so each lane loads its own
// contiguous run of K and the B fragment is built from the same run.
//
// Int4 tiles compute, per 64-group, P = X . (128 + q) with q turned into the
// bf16 value 128+q by one bit-or (0x4300 | q), the group sum Sx = X . 1 by one
// more mma with an all-ones A, and fold the zero point and the scale in fp32:
// Y += s * (P - (128 + z) * Sx).  This is (q - z) * s without rounding the
// dequantised weight to bf16 first.
//
// A CTA owns NT row tiles (16 rows each) over the whole K; its WK warps split
// K and their partial sums meet in shared memory in a fixed order, so results
// are deterministic and no global scratch is needed.
#pragma once
#include "common.cuh"

namespace sub {

enum GemvEpi : int {
  EPI_BF16 = 0,    // Y bf16 [M, ldy]
  EPI_F32 = 1,     // Y fp32 [M, ldy]
  EPI_RESID = 2,   // R fp32 [M, ldy] += acc
  EPI_GLU = 3,     // Y bf16 [M, ldy] = silu(gate) * up; segments 0 (gate) and 1 (up)
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
};

// Launch: int4 (is_w4) or bf16 weights, epilogue, M <= 16.
int32_t launch_gemv(const GemvArgs& a, bool is_w4, int epi, cudaStream_t stream);

}  // namespace sub
