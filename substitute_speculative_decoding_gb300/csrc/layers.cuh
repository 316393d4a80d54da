// Elementwise and row kernels of the decoder layer: embedding gather into the
// fp32 residual stream, RMSNorm to a bf16 matmul input, and the q/k/v epilogue
// (RoPE on q and k, bf16 rounding, K/V written into the paged cache).
#pragma once
#include "common.cuh"

namespace sub {

struct RowSet {
  // row r carries token tokens[r] (or tree.token[slot0 + r]) at position
  // base + depth[r]; its K/V go to cache position tree_base + slot0 + r.
  const int32_t* tokens;
  const int32_t* depth;      // [rows] or null (chain: depth = slot0 + r)
  int slot0;
  int64_t base;              // position of slot 0 ...
  const int32_t* base_dev;   // ... or read on the device
};

// ss_out non-null: factored RMSNorm (xn = bf16(x * gain), ss_out[r] = sum of
// x[r]^2, one part of the consumer's RowScale).
int32_t launch_embed(const uint16_t* embed, int hidden, const RowSet& rs, int rows, float* x,
                     const uint16_t* gain, float eps, uint16_t* xn, float* ss_out, cudaStream_t st);
// Rows entering a forward at a later layer: x = src, xn (and ss_out) as launch_embed forms them.
int32_t launch_rows_in(const float* src, int hidden, int rows, float* x, const uint16_t* gain,
                       float eps, uint16_t* xn, float* ss_out, cudaStream_t st);
// dst = x for rows x hidden floats (the residual stream handed to a later forward).
int32_t launch_rows_out(const float* x, int hidden, int rows, float* dst, cudaStream_t st);
int32_t launch_rmsnorm(const float* x, const uint16_t* gain, int rows, int hidden, float eps,
                       uint16_t* out, cudaStream_t st);

struct QkvPostArgs {
  const float* qkv;          // [rows, (Hq + 2 Hkv) * D] fp32
  int rows, n_heads_q, n_heads_kv, head_dim;
  const float2* rope;        // [max_pos, D/2] (cos, sin)
  int max_pos;
  RowSet rs;
  uint16_t* q_out;           // [rows, Hq, D] bf16
  uint16_t* k_cache;
  uint16_t* v_cache;
  const int32_t* page_table;
  int page_size, n_pages, layer;
};
int32_t launch_qkv_post(const QkvPostArgs& a, cudaStream_t st);

}  // namespace sub
