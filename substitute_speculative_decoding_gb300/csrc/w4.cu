// Int4 substitute construction: group-64 min-max pack and dequant.
//
// The draft's substitute layers are data-free 4-bit copies of the offloaded
// target layers ("SubSpec: Using the Target Model's Own Low-Bit Shadow as Its
// Draft Model", 2.2 Step 4; "Speculate Deep and Accurate" card, Approach).
// Quantiser (per row and 64-element group along K, all steps single IEEE fp32
// operations, no fast-math):
//   s = bf16((hi - lo) / 15), s = 1 if that rounds to 0;  z = bf16(-lo / s)
//   q = clamp(rint(w / s + z), 0, 15);   deq = bf16((q - z) * s)
// One warp owns one (row, group): lane l holds elements 2l, 2l+1 and writes
// byte l of the group (element 2l in the low nibble).
#include "common.cuh"

namespace sub {

__global__ void w4_pack_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                               uint8_t* __restrict__ q, uint16_t* __restrict__ scale,
                               uint16_t* __restrict__ zero) {
  const int64_t G = (K + 63) / 64;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (warp >= N * G) return;
  const int64_t row = warp / G, g = warp % G;
  const int64_t k = g * 64 + 2 * lane;
  const bool valid = k < K;  // K % 8 == 0: both elements of the pair agree
  float w0 = 0.f, w1 = 0.f;
  if (valid) {
    uint32_t pair = *reinterpret_cast<const uint32_t*>(W + row * K + k);
    w0 = bf16lo(pair);
    w1 = bf16hi(pair);
  }
  float lo = valid ? fminf(w0, w1) : INFINITY;
  float hi = valid ? fmaxf(w0, w1) : -INFINITY;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
  uint16_t sb = f32_to_bf16_bits(s32);
  float s = bf16_bits_to_f32(sb);
  if (s == 0.0f) { s = 1.0f; sb = 0x3f80; }
  const uint16_t zb = f32_to_bf16_bits(__fdiv_rn(-lo, s));
  const float z = bf16_bits_to_f32(zb);
  uint32_t c0 = 0, c1 = 0;
  if (valid) {
    c0 = (uint32_t)fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(w0, s), z)), 0.f), 15.f);
    c1 = (uint32_t)fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(w1, s), z)), 0.f), 15.f);
  }
  q[row * G * 32 + g * 32 + lane] = (uint8_t)(c0 | (c1 << 4));
  if (lane == 0) {
    scale[row * G + g] = sb;
    zero[row * G + g] = zb;
  }
}

__global__ void w4_dequant_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ scale,
                                  const uint16_t* __restrict__ zero, int64_t N, int64_t K,
                                  uint16_t* __restrict__ out) {
  const int64_t G = (K + 63) / 64;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // one byte = 2 elements
  if (i >= N * G * 32) return;
  const int64_t row = i / (G * 32), rem = i % (G * 32);
  const int64_t g = rem / 32;
  const int64_t k = g * 64 + 2 * (rem % 32);
  if (k >= K) return;
  const uint8_t b = q[i];
  const float s = bf16_bits_to_f32(scale[row * G + g]);
  const float z = bf16_bits_to_f32(zero[row * G + g]);
  // (q - z) and its product with s are exact in fp32; one rounding to bf16.
  const float d0 = __fmul_rn(__fsub_rn((float)(b & 15), z), s);
  const float d1 = __fmul_rn(__fsub_rn((float)(b >> 4), z), s);
  *reinterpret_cast<uint32_t*>(out + row * K + k) = pack_bf16x2(d0, d1);
}

int32_t w4_check(int64_t N, int64_t K, int32_t group) {
  if (group != 64) return fail(SUB_EUNSUPPORTED, "group must be 64");
  SUB_CHECK_ARG(N >= 1 && K >= 1, "N and K must be positive");
  SUB_CHECK_ARG(K % 8 == 0, "K must be a multiple of 8 (16-byte rows)");
  return SUB_OK;
}

}  // namespace sub

using namespace sub;

extern "C" int32_t sub_w4_pack(const sub_bf16* W, int64_t N, int64_t K, int32_t group,
                               uint8_t* q, sub_bf16* scale, sub_bf16* zero, void* stream) {
  SUB_TRY(w4_check(N, K, group));
  SUB_CHECK_ARG(W && q && scale && zero, "null pointer");
  SUB_CHECK_ARG(aligned16(W), "W must be 16-byte aligned");
  const int64_t warps = N * ((K + 63) / 64);
  const int threads = 256;
  const int64_t blocks = cdiv(warps, threads / 32);
  SUB_CHECK_ARG(blocks < (1ll << 31), "matrix too large");
  w4_pack_kernel<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(W, N, K, q, scale, zero);
  return check_launch("w4_pack");
}

extern "C" int32_t sub_w4_dequant(const uint8_t* q, const sub_bf16* scale, const sub_bf16* zero,
                                  int64_t N, int64_t K, int32_t group, sub_bf16* W_out,
                                  void* stream) {
  SUB_TRY(w4_check(N, K, group));
  SUB_CHECK_ARG(W_out && q && scale && zero, "null pointer");
  SUB_CHECK_ARG(aligned16(W_out), "W_out must be 16-byte aligned");
  const int64_t bytes = N * ((K + 63) / 64) * 32;
  const int threads = 256;
  const int64_t blocks = cdiv(bytes, threads);
  SUB_CHECK_ARG(blocks < (1ll << 31), "matrix too large");
  w4_dequant_kernel<<<(unsigned)blocks, threads, 0, as_stream(stream)>>>(q, scale, zero, N, K,
                                                                          W_out);
  return check_launch("w4_dequant");
}
