// Shared device/host helpers of the SubSpec library (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string>
#include <cstring>
#include "../../include/sub_api.h"

namespace sub {

// ---------------------------------------------------------------- errors --
void set_error(const std::string& msg);
int32_t fail(int32_t code, const std::string& msg);
int32_t check_launch(const char* what);

#define SUB_CHECK_ARG(cond, msg) \
  do { if (!(cond)) return ::sub::fail(SUB_EINVAL, msg); } while (0)
#define SUB_CUDA_TRY(expr) \
  do { cudaError_t _e = (expr); if (_e != cudaSuccess) \
    return ::sub::fail(SUB_ECUDA, std::string(#expr) + ": " + cudaGetErrorString(_e)); } while (0)
#define SUB_TRY(expr) do { int32_t _s = (expr); if (_s != SUB_OK) return _s; } while (0)

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ------------------------------------------- programmatic dependent launch --
// Kernels of the decode path are launched with programmatic stream
// serialisation: the next kernel may start while this one drains.  Every such
// kernel calls pdl_wait() before it touches anything an earlier kernel wrote
// (weights may be read before the wait), and signals pdl_trigger() only from
// threads that have passed their own pdl_wait().  By induction, when a kernel
// starts, every kernel before its immediate predecessor has finished; the
// attention kernel's reads ahead of its wait rely on exactly this.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

bool pdl_enabled();   // SUB_PDL=0 in the environment turns it off
bool env_flag(const char* name, bool dflt);
// Host-side fault injection (SUB_FAULT, read at each call): true when the
// environment asks the `index`-th event of `kind` ("alloc" with "alloc:N",
// "h2d" for every streamed copy) to fail.
bool fault_injected(const char* kind, int index);

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ bf16 bits --
__host__ __device__ inline float bf16_bits_to_f32(uint16_t b) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(((uint32_t)b) << 16);
#else
  uint32_t u = ((uint32_t)b) << 16; float f; memcpy(&f, &u, 4); return f;
#endif
}

// Round-to-nearest-even fp32 -> bf16 bits (finite values).
__device__ inline uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Two fp32 -> packed bf16x2 (lo = a, hi = b), round to nearest even.
__device__ inline uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ inline float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ inline float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------- mma.sync --
// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulators.
__device__ inline void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                      uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ inline uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ inline uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ inline uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ inline float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}
// 64-bit ranking key: larger value first, then smaller index.
__device__ inline unsigned long long rank_key(float v, uint32_t idx) {
  return ((unsigned long long)float_key(v) << 32) | (unsigned long long)(0xffffffffu - idx);
}
__device__ inline uint32_t rank_idx(unsigned long long k) {
  return 0xffffffffu - (uint32_t)(k & 0xffffffffull);
}

}  // namespace sub
