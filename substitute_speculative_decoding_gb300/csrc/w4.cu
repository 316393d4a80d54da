// Low-bit substitute construction: group-64 min-max pack and dequant for
// 4-bit codes (the pages' substitutes) and 2- or 3-bit codes (the lower and
// mixed precisions they leave open).
//
// The draft's substitute layers are data-free low-bit copies of the offloaded
// target layers ("SubSpec: Using the Target Model's Own Low-Bit Shadow as Its
// Draft Model", 2.2 Step 4, 5.1 point 2, 10.1 (2); "Speculate Deep and
// Accurate" card, Approach).  Quantiser with L = 2^bits - 1 levels (per row
// and 64-element group along K, all steps single IEEE fp32 operations, no
// fast-math):
//   s = bf16((hi - lo) / L), s = 1 if that rounds to 0;  z = bf16(-lo / s)
//   q = clamp(rint(w / s + z), 0, L);   deq = bf16((q - z) * s)
// Code layout of a group (8 * bits bytes):
//   4 bits: byte j = element 2j (low nibble) | element 2j+1 << 4
//   2 bits: byte j = elements 4j .. 4j+3 at bits 0-1, 2-3, 4-5, 6-7
//   3 bits: bytes 0..15 the 2-bit layout of (q & 3); bit i of byte 16 + j is
//           q(8j + i) >> 2
// HQQ zero optimisation (sub_wq_pack_hqq; the pages' quantiser, "Low-Bit
// Shadow" report Critique 3 and 6.2, restated from the published
// half-quadratic method): the min-max scale is kept and the zero refined by
// `iters` steps of  q = clamp(rint(w/s + z), 0, L),  r = w - s (q - z),
// e = sign(r) max(|r| - |r|^(-1/2) / beta, 0),  z = mean(q - (w - e)/s),
// beta *= 1.01 (beta starts at 10); the zero with the smallest sum |r| is kept,
// rounded to bf16, and the codes formed with it.
// One warp owns one (row, group): lane l holds elements 2l and 2l + 1.
#include "common.cuh"

namespace sub {

// Codes c0 (element 2 lane) and c1 (element 2 lane + 1) of every lane into
// the group's bytes (layouts above).  All 32 lanes call it.
template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t* grp, int lane, uint32_t c0, uint32_t c1) {
  if constexpr (BITS == 4) {
    grp[lane] = (uint8_t)(c0 | (c1 << 4));
  } else {
    // low two bits: lanes 2j and 2j + 1 make byte j
    const uint32_t pair = (c0 & 3u) | ((c1 & 3u) << 2);
    const uint32_t next = __shfl_down_sync(0xffffffffu, pair, 1);
    if ((lane & 1) == 0) grp[lane >> 1] = (uint8_t)(pair | (next << 4));
    if constexpr (BITS == 3) {
      // high bits: element e = 2l + t has its bit in ballot t at position l
      const uint32_t m0 = __ballot_sync(0xffffffffu, (c0 >> 2) & 1u);
      const uint32_t m1 = __ballot_sync(0xffffffffu, (c1 >> 2) & 1u);
      if (lane < 8) {
        uint32_t byte = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t m = (i & 1) ? m1 : m0;
          byte |= ((m >> (4 * lane + (i >> 1))) & 1u) << i;
        }
        grp[16 + lane] = (uint8_t)byte;
      }
    }
  }
}

// Sum over the group's 64 entries (two per lane) in one fixed order:
// a = x0 + x1 per lane, then a += a of lane (l xor o), o = 16, 8, 4, 2, 1.
// Every lane returns the same value.
__device__ __forceinline__ float pair_sum64(float x0, float x1) {
  float a = __fadd_rn(x0, x1);
#pragma unroll
  for (int o = 16; o; o >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

__device__ __forceinline__ float code_for(float w, float s, float z, float levels) {
  return fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(w, s), z)), 0.f), levels);
}

// HQQ zero optimisation of one group (see hqq_iters in sub_wq_pack_hqq):
// min-max scale fixed, zero refined by half-quadratic steps with p = 1/2,
// the zero with the smallest sum |w - s (q - z)| kept.  Every operation is
// one correctly rounded fp32 operation (no contraction into FMA).
__device__ float hqq_zero(float w0, float w1, bool v0, bool v1, int cnt, float s, float z0,
                          float levels, int iters, float beta0, float kappa) {
  float z = z0, best_z = z0, best_err = 0.f, beta = beta0;
  for (int it = 0; it < iters; ++it) {
    const float q0 = code_for(w0, s, z, levels), q1 = code_for(w1, s, z, levels);
    const float r0 = v0 ? __fsub_rn(w0, __fmul_rn(s, __fsub_rn(q0, z))) : 0.f;
    const float r1 = v1 ? __fsub_rn(w1, __fmul_rn(s, __fsub_rn(q1, z))) : 0.f;
    const float err = pair_sum64(fabsf(r0), fabsf(r1));
    if (it == 0 || err < best_err) {
      best_err = err;
      best_z = z;
    }
    // shrinkage: sign(r) max(|r| - (1 / sqrt|r|) / beta, 0); 0 at r = 0
    auto shrink = [&](float r) {
      const float ar = fabsf(r);
      if (ar == 0.f) return 0.f;
      const float th = __fdiv_rn(__fdiv_rn(1.f, __fsqrt_rn(ar)), beta);
      return copysignf(fmaxf(__fsub_rn(ar, th), 0.f), r);
    };
    const float e0 = shrink(r0), e1 = shrink(r1);
    const float t0 = v0 ? __fsub_rn(q0, __fdiv_rn(__fsub_rn(w0, e0), s)) : 0.f;
    const float t1 = v1 ? __fsub_rn(q1, __fdiv_rn(__fsub_rn(w1, e1), s)) : 0.f;
    z = __fdiv_rn(pair_sum64(t0, t1), (float)cnt);
    beta = __fmul_rn(beta, kappa);
  }
  return best_z;
}

// iters == 0: the min-max quantiser; iters >= 1: HQQ zero optimisation.
template <int BITS>
__global__ void wq_pack_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                               uint8_t* __restrict__ q, uint16_t* __restrict__ scale,
                               uint16_t* __restrict__ zero, int iters, float beta0, float kappa) {
  constexpr int GB = 8 * BITS;                 // bytes per group
  constexpr float LEVELS = (float)((1 << BITS) - 1);
  const int64_t G = (K + 63) / 64;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (warp >= N * G) return;   // uniform per warp
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
  const float s32 = __fdiv_rn(__fsub_rn(hi, lo), LEVELS);
  uint16_t sb = f32_to_bf16_bits(s32);
  float s = bf16_bits_to_f32(sb);
  if (s == 0.0f) { s = 1.0f; sb = 0x3f80; }
  float zf = __fdiv_rn(-lo, s);
  if (iters > 0) {
    const int cnt = (int)(K - g * 64 < 64 ? K - g * 64 : 64);
    zf = hqq_zero(w0, w1, valid, valid, cnt, s, zf, LEVELS, iters, beta0, kappa);
  }
  const uint16_t zb = f32_to_bf16_bits(zf);
  const float z = bf16_bits_to_f32(zb);
  uint32_t c0 = 0, c1 = 0;
  if (valid) {
    c0 = (uint32_t)code_for(w0, s, z, LEVELS);
    c1 = (uint32_t)code_for(w1, s, z, LEVELS);
  }
  store_codes<BITS>(q + row * G * GB + g * GB, lane, c0, c1);
  if (lane == 0) {
    scale[row * G + g] = sb;
    zero[row * G + g] = zb;
  }
}

// Code of element j (0..63) of a group.
template <int BITS>
__device__ __forceinline__ uint32_t code_of(const uint8_t* grp, int j) {
  if constexpr (BITS == 4) return (grp[j >> 1] >> (4 * (j & 1))) & 15u;
  uint32_t c = (grp[j >> 2] >> (2 * (j & 3))) & 3u;
  if constexpr (BITS == 3) c |= ((grp[16 + (j >> 3)] >> (j & 7)) & 1u) << 2;
  return c;
}

template <int BITS>
__global__ void wq_dequant_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ scale,
                                  const uint16_t* __restrict__ zero, int64_t N, int64_t K,
                                  uint16_t* __restrict__ out) {
  constexpr int GB = 8 * BITS;
  const int64_t G = (K + 63) / 64;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // one element pair
  if (i >= N * G * 32) return;
  const int64_t row = i / (G * 32), rem = i % (G * 32);
  const int64_t g = rem / 32;
  const int j = 2 * (int)(rem % 32);
  const int64_t k = g * 64 + j;
  if (k >= K) return;
  const uint8_t* grp = q + row * G * GB + g * GB;
  const float s = bf16_bits_to_f32(scale[row * G + g]);
  const float z = bf16_bits_to_f32(zero[row * G + g]);
  // (q - z) and its product with s are exact in fp32; one rounding to bf16.
  const float d0 = __fmul_rn(__fsub_rn((float)code_of<BITS>(grp, j), z), s);
  const float d1 = __fmul_rn(__fsub_rn((float)code_of<BITS>(grp, j + 1), z), s);
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

static int32_t wq_pack(const sub_bf16* W, int64_t N, int64_t K, int32_t group, int32_t bits,
                       uint8_t* q, sub_bf16* scale, sub_bf16* zero, void* stream,
                       int32_t iters = 0) {
  SUB_TRY(w4_check(N, K, group));
  SUB_CHECK_ARG(iters >= 0 && iters <= 1000, "iters must be in [0, 1000]");
  const float beta0 = 10.0f, kappa = 1.01f;
  SUB_CHECK_ARG(bits == 2 || bits == 3 || bits == 4, "bits must be 2, 3 or 4");
  SUB_CHECK_ARG(W && q && scale && zero, "null pointer");
  SUB_CHECK_ARG(aligned16(W), "W must be 16-byte aligned");
  const int64_t warps = N * ((K + 63) / 64);
  const int threads = 256;
  const int64_t blocks = cdiv(warps, threads / 32);
  SUB_CHECK_ARG(blocks < (1ll << 31), "matrix too large");
  const cudaStream_t st = as_stream(stream);
  if (bits == 4)
    wq_pack_kernel<4><<<(unsigned)blocks, threads, 0, st>>>(W, N, K, q, scale, zero, iters, beta0,
                                                              kappa);
  if (bits == 3)
    wq_pack_kernel<3><<<(unsigned)blocks, threads, 0, st>>>(W, N, K, q, scale, zero, iters, beta0,
                                                              kappa);
  if (bits == 2)
    wq_pack_kernel<2><<<(unsigned)blocks, threads, 0, st>>>(W, N, K, q, scale, zero, iters, beta0,
                                                              kappa);
  return check_launch("wq_pack");
}

static int32_t wq_dequant(const uint8_t* q, const sub_bf16* scale, const sub_bf16* zero,
                          int64_t N, int64_t K, int32_t group, int32_t bits, sub_bf16* W_out,
                          void* stream) {
  SUB_TRY(w4_check(N, K, group));
  SUB_CHECK_ARG(bits == 2 || bits == 3 || bits == 4, "bits must be 2, 3 or 4");
  SUB_CHECK_ARG(W_out && q && scale && zero, "null pointer");
  SUB_CHECK_ARG(aligned16(W_out), "W_out must be 16-byte aligned");
  const int64_t pairs = N * ((K + 63) / 64) * 32;
  const int threads = 256;
  const int64_t blocks = cdiv(pairs, threads);
  SUB_CHECK_ARG(blocks < (1ll << 31), "matrix too large");
  const cudaStream_t st = as_stream(stream);
  if (bits == 4)
    wq_dequant_kernel<4><<<(unsigned)blocks, threads, 0, st>>>(q, scale, zero, N, K, W_out);
  if (bits == 3)
    wq_dequant_kernel<3><<<(unsigned)blocks, threads, 0, st>>>(q, scale, zero, N, K, W_out);
  if (bits == 2)
    wq_dequant_kernel<2><<<(unsigned)blocks, threads, 0, st>>>(q, scale, zero, N, K, W_out);
  return check_launch("wq_dequant");
}

extern "C" int32_t sub_w4_pack(const sub_bf16* W, int64_t N, int64_t K, int32_t group,
                               uint8_t* q, sub_bf16* scale, sub_bf16* zero, void* stream) {
  return wq_pack(W, N, K, group, 4, q, scale, zero, stream);
}

extern "C" int32_t sub_w4_dequant(const uint8_t* q, const sub_bf16* scale, const sub_bf16* zero,
                                  int64_t N, int64_t K, int32_t group, sub_bf16* W_out,
                                  void* stream) {
  return wq_dequant(q, scale, zero, N, K, group, 4, W_out, stream);
}

extern "C" int32_t sub_wq_pack(const sub_bf16* W, int64_t N, int64_t K, int32_t group,
                               int32_t bits, uint8_t* q, sub_bf16* scale, sub_bf16* zero,
                               void* stream) {
  return wq_pack(W, N, K, group, bits, q, scale, zero, stream);
}

extern "C" int32_t sub_wq_dequant(const uint8_t* q, const sub_bf16* scale, const sub_bf16* zero,
                                  int64_t N, int64_t K, int32_t group, int32_t bits,
                                  sub_bf16* W_out, void* stream) {
  return wq_dequant(q, scale, zero, N, K, group, bits, W_out, stream);
}

extern "C" int32_t sub_wq_pack_hqq(const sub_bf16* W, int64_t N, int64_t K, int32_t group,
                                   int32_t bits, int32_t iters, uint8_t* q, sub_bf16* scale,
                                   sub_bf16* zero, void* stream) {
  SUB_CHECK_ARG(iters >= 1, "iters must be >= 1");
  return wq_pack(W, N, K, group, bits, q, scale, zero, stream, iters);
}
