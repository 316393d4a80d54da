// Row kernels of the decoder layer (see layers.cuh).  The residual stream is
// fp32; matmul inputs and the KV cache are bf16, rounded to nearest even.
#include "layers.cuh"

namespace sub {

__device__ __forceinline__ int row_depth(const RowSet& rs, int r) {
  return rs.depth ? rs.depth[r] : rs.slot0 + r;
}
__device__ __forceinline__ int64_t row_base(const RowSet& rs) {
  return rs.base_dev ? (int64_t)*rs.base_dev : rs.base;
}

// x[r] = embed[token[r]] (fp32 residual) and the first layer's matmul input:
// xn[r] = bf16(RMSNorm(x[r]) * gain), or, factored (ss non-null),
// xn[r] = bf16(x[r] * gain) and ss[r] = sum of x[r]^2, the single part from
// which the consumer forms the row scale rsqrt(ss / hidden + eps).  One CTA per row.
__global__ void embed_kernel(const uint16_t* __restrict__ embed, int hidden, RowSet rs,
                             float* __restrict__ x, const uint16_t* __restrict__ gain, float eps,
                             uint16_t* __restrict__ xn, float* __restrict__ ss_out) {
  __shared__ float s_part[32];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int64_t tok = rs.tokens[r];
  const uint16_t* src = embed + tok * hidden;
  float ss = 0.f;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) {
    const float v = bf16_bits_to_f32(src[i]);
    x[(int64_t)r * hidden + i] = v;
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_part[w];
  const float inv = rsqrtf(tot / (float)hidden + eps);
  if (ss_out && threadIdx.x == 0) ss_out[r] = tot;
  const float scale = ss_out ? 1.0f : inv;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x)
    reinterpret_cast<__nv_bfloat16*>(xn)[(int64_t)r * hidden + i] =
        __float2bfloat16_rn(bf16_bits_to_f32(src[i]) * scale * bf16_bits_to_f32(gain[i]));
}

int32_t launch_embed(const uint16_t* embed, int hidden, const RowSet& rs, int rows, float* x,
                     const uint16_t* gain, float eps, uint16_t* xn, float* ss_out, cudaStream_t st) {
  if (rows <= 0) return SUB_OK;
  SUB_CUDA_TRY(launch_k(embed_kernel, dim3(rows), dim3(256), 0, st, embed, hidden, rs, x, gain,
                        eps, xn, ss_out));
  return SUB_OK;
}

// Rows that enter a forward part-way (the verify from a layer the draft has
// already computed for the same nodes): x = src row, and the first layer's
// RMSNorm input exactly as embed_kernel forms it from an embedding row.
__global__ void rows_in_kernel(const float* __restrict__ src, int hidden,
                               float* __restrict__ x, const uint16_t* __restrict__ gain, float eps,
                               uint16_t* __restrict__ xn, float* __restrict__ ss_out) {
  __shared__ float s_part[32];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const float* sr = src + (int64_t)r * hidden;
  float ss = 0.f;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) {
    const float v = sr[i];
    x[(int64_t)r * hidden + i] = v;
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_part[w];
  const float inv = rsqrtf(tot / (float)hidden + eps);
  if (ss_out && threadIdx.x == 0) ss_out[r] = tot;
  const float scale = ss_out ? 1.0f : inv;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x)
    reinterpret_cast<__nv_bfloat16*>(xn)[(int64_t)r * hidden + i] =
        __float2bfloat16_rn(sr[i] * scale * bf16_bits_to_f32(gain[i]));
}

int32_t launch_rows_in(const float* src, int hidden, int rows, float* x, const uint16_t* gain,
                       float eps, uint16_t* xn, float* ss_out, cudaStream_t st) {
  if (rows <= 0) return SUB_OK;
  SUB_CUDA_TRY(launch_k(rows_in_kernel, dim3(rows), dim3(256), 0, st, src, hidden, x, gain, eps,
                        xn, ss_out));
  return SUB_OK;
}

// dst[r, :] = x[r, :] for `rows` rows of `hidden` floats (16-byte aligned rows).
__global__ void rows_out_kernel(const float4* __restrict__ x, int n4, float4* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n4) dst[i] = x[i];
}

int32_t launch_rows_out(const float* x, int hidden, int rows, float* dst, cudaStream_t st) {
  if (rows <= 0) return SUB_OK;
  SUB_CHECK_ARG(hidden % 4 == 0 && aligned16(x) && aligned16(dst), "rows_out: alignment");
  const int n4 = rows * hidden / 4;
  SUB_CUDA_TRY(launch_k(rows_out_kernel, dim3((n4 + 255) / 256), dim3(256), 0, st,
                        reinterpret_cast<const float4*>(x), n4, reinterpret_cast<float4*>(dst)));
  return SUB_OK;
}

// y = bf16(x * rsqrt(mean(x^2) + eps) * gain); one CTA per row, fixed-order sum.
__global__ void rmsnorm_kernel(const float* __restrict__ x, const uint16_t* __restrict__ gain,
                               int hidden, float eps, uint16_t* __restrict__ out) {
  __shared__ float s_part[32];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const float* xr = x + (int64_t)r * hidden;
  float ss = 0.f;
  for (int i = threadIdx.x; i < hidden; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_part[w];
  const float inv = rsqrtf(tot / (float)hidden + eps);
  for (int i = threadIdx.x; i < hidden; i += blockDim.x)
    reinterpret_cast<__nv_bfloat16*>(out)[(int64_t)r * hidden + i] =
        __float2bfloat16_rn(xr[i] * inv * bf16_bits_to_f32(gain[i]));
}

int32_t launch_rmsnorm(const float* x, const uint16_t* gain, int rows, int hidden, float eps,
                       uint16_t* out, cudaStream_t st) {
  if (rows <= 0) return SUB_OK;
  SUB_CUDA_TRY(launch_k(rmsnorm_kernel, dim3(rows), dim3(256), 0, st, x, gain, hidden, eps, out));
  return SUB_OK;
}

// One CTA per row: q heads get RoPE -> bf16 q_out; k heads RoPE -> cache;
// v heads -> cache.  Rotate-half pairing: element i with i + D/2.
__global__ void qkv_post_kernel(QkvPostArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int D = a.head_dim, half = D / 2;
  const int nh = a.n_heads_q + 2 * a.n_heads_kv;
  const int64_t base = row_base(a.rs);
  const int64_t pos = base + row_depth(a.rs, r);
  const int64_t kvpos = base + a.rs.slot0 + r;
  const float* src = a.qkv + (int64_t)r * nh * D;
  const float2* cs = a.rope + (pos < a.max_pos ? pos : a.max_pos - 1) * half;
  const size_t head_stride = (size_t)a.page_size * D;
  const size_t page_stride = (size_t)a.n_heads_kv * head_stride;
  const size_t slot_off = (size_t)a.layer * a.n_pages * page_stride +
                          (size_t)a.page_table[kvpos / a.page_size] * page_stride +
                          (size_t)(kvpos % a.page_size) * D;
  for (int idx = threadIdx.x; idx < nh * half; idx += blockDim.x) {
    const int h = idx / half, i = idx % half;
    const float x1 = src[h * D + i], x2 = src[h * D + i + half];
    if (h < a.n_heads_q + a.n_heads_kv) {
      const float2 c = cs[i];
      const float y1 = x1 * c.x - x2 * c.y;
      const float y2 = x2 * c.x + x1 * c.y;
      if (h < a.n_heads_q) {
        uint16_t* q = a.q_out + ((int64_t)r * a.n_heads_q + h) * D;
        q[i] = f32_to_bf16_bits(y1);
        q[i + half] = f32_to_bf16_bits(y2);
      } else {
        uint16_t* k = a.k_cache + slot_off + (size_t)(h - a.n_heads_q) * head_stride;
        k[i] = f32_to_bf16_bits(y1);
        k[i + half] = f32_to_bf16_bits(y2);
      }
    } else {
      uint16_t* v = a.v_cache + slot_off + (size_t)(h - a.n_heads_q - a.n_heads_kv) * head_stride;
      v[i] = f32_to_bf16_bits(x1);
      v[i + half] = f32_to_bf16_bits(x2);
    }
  }
}

int32_t launch_qkv_post(const QkvPostArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return SUB_OK;
  SUB_CUDA_TRY(launch_k(qkv_post_kernel, dim3(a.rows), dim3(256), 0, st, a));
  return SUB_OK;
}

}  // namespace sub
