// Tiled tensor-core GEMM for tree-shaped products (M > 16 rows): the verify
// pass over every tree node, the prefill, and int4 products at tree widths.
// Y[m, n] = sum_k X[m, k] W[n, k]; rows are independent (no split over K that
// depends on M), so a row's result does not depend on how many rows share
// the pass.
#pragma once
#include "gemv.cuh"

namespace sub {

int32_t gemm_init();
// Same argument block and epilogues as the GEMV (GemvArgs); M is unbounded.
int32_t launch_gemm(const GemvArgs& a, bool is_w4, int epi, cudaStream_t stream);

// Tensor-core (tcgen05, TMEM accumulator, TMA-fed) variant for bf16 weights
// and the bf16/f32/residual/SiLU-GLU epilogues (gemm_tc.cu).  Launches and sets
// *done when the product suits it; launch_gemm tries it first (SUB_GEMM_TC=0
// turns it off).  Split-K partials use split_part / split_cnt.
int32_t launch_gemm_tc(const GemvArgs& a, bool is_w4, int epi, cudaStream_t stream, bool* done);
int32_t gemm_tc_init();
size_t gemm_tc_scratch_floats(const GemvArgs& a, bool is_w4, int epi);
int32_t gemm_tc_timeouts(unsigned int* out);

// Dispatch on M: GEMV for M <= 16, tiled GEMM otherwise, except int4 products
// with a bf16 output up to 32 rows, which take the TMA GEMV's four token tiles.
// 2- and 3-bit codes have the GEMV only (the draft's tree levels, M <= 16).
inline int32_t launch_matmul(const GemvArgs& a, bool is_w4, int epi, cudaStream_t stream) {
  if (a.M <= 16) return launch_gemv(a, is_w4, epi, stream);
  if (is_w4 && code_bits(a) != 4)
    return fail(SUB_EUNSUPPORTED, "2- and 3-bit weights: M must be <= 16 here");
  if (is_w4 && a.M <= 32 && epi == EPI_BF16) {
    // up to 32 rows the TMA GEMV with four token tiles beats the tensor-core
    // GEMM on an int4 product, where its plan and scratch fit
    bool done = false;
    SUB_TRY(launch_gemv_tma(a, true, epi, stream, &done));
    if (done) return SUB_OK;
  }
  return launch_gemm(a, is_w4, epi, stream);
}

}  // namespace sub
