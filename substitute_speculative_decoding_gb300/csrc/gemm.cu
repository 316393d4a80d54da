// Tiled GEMM on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with a 3-stage
// cp.async pipeline: CTA tile 128 x 128 x 64, eight warps of 64 x 32.  The
// activation tile streams with cp.async; the weight tile streams with
// cp.async (bf16) or is dequantised from packed int4 into shared memory with
// the exact rule bf16((q - z) * s).  Shared tiles use a 128-byte row with the
// 16-byte chunk index XOR-swizzled by (row & 7), so ldmatrix is conflict-free.
// The epilogue stages the fp32 tile in shared memory and writes coalesced rows.
#include <mutex>
#include "gemm.cuh"

namespace sub {

namespace {
constexpr int BM = 128, BN = 128, BK = 64, STAGES = 3, THREADS = 256;
constexpr int TILE_BYTES = BM * BK * 2;  // 16 KB per operand per stage
constexpr int SMEM_BYTES = STAGES * 2 * TILE_BYTES;  // 96 KB
constexpr int EPI_LD = BN + 4;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ int swz(int row, int chunk) { return row * 8 + (chunk ^ (row & 7)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ float silu_g(float x) { return x / (1.0f + expf(-x)); }

// Row n of the stacked weight segments -> (segment, local row); n < total rows.
__device__ __forceinline__ int seg_of(const GemvArgs& a, int n, int& local) {
  int s = 0, start = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (s < a.n_seg - 1 && n >= a.seg_end[s]) { start = a.seg_end[s]; ++s; }
  local = n - start;
  return s;
}
}  // namespace

template <bool W4, int EPI>
__global__ void __launch_bounds__(THREADS) gemm_kernel(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool GLU = (EPI == EPI_GLU);
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;
  const int m0 = blockIdx.y * BM;
  // GLU: output columns [c0, c0+64); B rows 0..63 from the gate, 64..127 from the up rows
  const int n0 = GLU ? blockIdx.x * (BN / 2) : blockIdx.x * BN;
  const int K = a.K;
  const int KT = (K + BK - 1) / BK;
  const int G = (K + 63) / 64;

  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * TILE_BYTES;

  // ---- per-thread load assignments ----
  // A: 4 chunks per thread: chunk c = tid + i*256 -> row c/8, kc c%8
  const uint16_t* a_src[4];
  bool a_ok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = tid + i * THREADS, r = c >> 3, kc = c & 7;
    const int m = m0 + r;
    a_ok[i] = m < a.M;
    a_src[i] = a.X + (int64_t)(a_ok[i] ? m : 0) * a.ldx + kc * 8;
  }
  // B (bf16): same chunk map over 128 weight rows
  const uint16_t* b_src[4];
  bool b_ok[4];
  // B (int4): thread -> (row tid/2, half tid%2)
  const uint8_t* q_src = nullptr;
  const uint16_t* s_src = nullptr;
  const uint16_t* z_src = nullptr;
  bool q_ok = false;
  if constexpr (!W4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = tid + i * THREADS, r = c >> 3, kc = c & 7;
      int seg, local;
      bool ok;
      if (GLU) {
        seg = r >> 6;
        local = n0 + (r & 63);
        ok = local < a.N;
      } else {
        const int n = n0 + r;
        ok = n < a.N;
        seg = seg_of(a, ok ? n : 0, local);
      }
      b_ok[i] = ok;
      b_src[i] = reinterpret_cast<const uint16_t*>(a.W[seg]) + (int64_t)(ok ? local : 0) * K + kc * 8;
    }
  } else {
    const int r = tid >> 1;
    int seg, local;
    if (GLU) {
      seg = r >> 6;
      local = n0 + (r & 63);
      q_ok = local < a.N;
    } else {
      const int n = n0 + r;
      q_ok = n < a.N;
      seg = seg_of(a, q_ok ? n : 0, local);
    }
    if (!q_ok) local = 0;
    q_src = reinterpret_cast<const uint8_t*>(a.W[seg]) + (int64_t)local * G * 32 + (tid & 1) * 16;
    s_src = a.S[seg] + (int64_t)local * G;
    z_src = a.Z[seg] + (int64_t)local * G;
  }

  auto load_a = [&](int stage, int kt) {
    const int k0 = kt * BK;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = tid + i * THREADS, r = c >> 3, kc = c & 7;
      const bool ok = a_ok[i] && (k0 + kc * 8 < K);
      cp_async16(smem_u32(sA + stage * TILE_BYTES + swz(r, kc) * 16), ok ? a_src[i] + k0 : a.X, ok);
    }
  };
  auto load_b16 = [&](int stage, int kt) {
    const int k0 = kt * BK;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = tid + i * THREADS, r = c >> 3, kc = c & 7;
      const bool ok = b_ok[i] && (k0 + kc * 8 < K);
      cp_async16(smem_u32(sB + stage * TILE_BYTES + swz(r, kc) * 16),
                 ok ? b_src[i] + k0 : reinterpret_cast<const uint16_t*>(a.W[0]), ok);
    }
  };
  // int4: registers for one k-tile (= one group) of this thread's half row
  auto fetch_q = [&](int kt, uint4& qv, uint16_t& sv, uint16_t& zv) {
    if (q_ok && kt < KT) {
      qv = __ldg(reinterpret_cast<const uint4*>(q_src + (int64_t)kt * 32));
      sv = __ldg(s_src + kt);
      zv = __ldg(z_src + kt);
    } else {
      qv = make_uint4(0, 0, 0, 0);
      sv = 0;
      zv = 0;
    }
  };
  auto store_q = [&](int stage, const uint4& qv, uint16_t sv, uint16_t zv) {
    const float s = bf16_bits_to_f32(sv), z = bf16_bits_to_f32(zv);
    const int r = tid >> 1, half = tid & 1;
    const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {   // chunk = 8 elements = one word of 8 nibbles
      const uint32_t w = words[c];
      uint32_t out[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {  // byte p: elements 2p (low nibble), 2p+1 (high)
        const float d0 = __fmul_rn(__fsub_rn((float)((w >> (8 * p)) & 15u), z), s);
        const float d1 = __fmul_rn(__fsub_rn((float)((w >> (8 * p + 4)) & 15u), z), s);
        out[p] = pack_bf16x2(d0, d1);
      }
      *reinterpret_cast<uint4*>(sB + stage * TILE_BYTES + swz(r, half * 4 + c) * 16) =
          make_uint4(out[0], out[1], out[2], out[3]);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

  // ---- prologue ----
  uint4 qv;
  uint16_t sv, zv;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) {
      load_a(s, s);
      if constexpr (!W4) load_b16(s, s);
      else {
        fetch_q(s, qv, sv, zv);
        store_q(s, qv, sv, zv);
      }
    }
    cp_commit();
  }

  for (int kt = 0; kt < KT; ++kt) {
    cp_wait<STAGES - 2>();
    __syncthreads();
    const int nk = kt + STAGES - 1;
    const int ns = nk % STAGES;
    if (nk < KT) {
      load_a(ns, nk);
      if constexpr (!W4) load_b16(ns, nk);
    }
    if constexpr (W4) fetch_q(nk, qv, sv, zv);
    cp_commit();

    const int st = kt % STAGES;
    const uint32_t aBase = smem_u32(sA + st * TILE_BYTES);
    const uint32_t bBase = smem_u32(sB + st * TILE_BYTES);
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t af[4][4], bfr[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = wm * 64 + i * 16 + (lane & 15);
        const int ch = kk * 2 + (lane >> 4);
        ldsm_x4(aBase + swz(r, ch) * 16, af[i][0], af[i][1], af[i][2], af[i][3]);
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int r = wn * 32 + jj * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = kk * 2 + ((lane >> 3) & 1);
        ldsm_x4(bBase + swz(r, ch) * 16, bfr[2 * jj][0], bfr[2 * jj][1], bfr[2 * jj + 1][0],
                bfr[2 * jj + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[i][j], af[i], bfr[j][0], bfr[j][1]);
    }
    if constexpr (W4) {
      if (nk < KT) store_q(ns, qv, sv, zv);
    }
  }
  cp_wait<0>();
  __syncthreads();

  // ---- epilogue through shared memory ----
  float* sC = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = wm * 64 + i * 16 + (lane >> 2);
      const int c = wn * 32 + j * 8 + 2 * (lane & 3);
      sC[r * EPI_LD + c] = acc[i][j][0];
      sC[r * EPI_LD + c + 1] = acc[i][j][1];
      sC[(r + 8) * EPI_LD + c] = acc[i][j][2];
      sC[(r + 8) * EPI_LD + c + 1] = acc[i][j][3];
    }
  __syncthreads();
  if constexpr (GLU) {
    for (int idx = tid; idx < BM * (BN / 2); idx += THREADS) {
      const int r = idx / (BN / 2), c = idx % (BN / 2);
      const int m = m0 + r, n = n0 + c;
      if (m >= a.M || n >= a.N) continue;
      const float gv = sC[r * EPI_LD + c], uv = sC[r * EPI_LD + c + 64];
      reinterpret_cast<__nv_bfloat16*>(a.Y)[(int64_t)m * a.ldy + n] =
          __float2bfloat16_rn(silu_g(gv) * uv);
    }
  } else {
    for (int idx = tid; idx < BM * BN; idx += THREADS) {
      const int r = idx / BN, c = idx % BN;
      const int m = m0 + r, n = n0 + c;
      if (m >= a.M || n >= a.N) continue;
      const float v = sC[r * EPI_LD + c];
      const int64_t o = (int64_t)m * a.ldy + n;
      if constexpr (EPI == EPI_BF16) reinterpret_cast<__nv_bfloat16*>(a.Y)[o] = __float2bfloat16_rn(v);
      else if constexpr (EPI == EPI_F32) reinterpret_cast<float*>(a.Y)[o] = v;
      else reinterpret_cast<float*>(a.Y)[o] += v;
    }
  }
}

// Opt every instantiation into 96 KB of dynamic shared memory once per process
// (before any stream capture: model creation calls this).
int32_t gemm_init() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    const void* ks[] = {
        (const void*)gemm_kernel<false, EPI_BF16>, (const void*)gemm_kernel<false, EPI_F32>,
        (const void*)gemm_kernel<false, EPI_RESID>, (const void*)gemm_kernel<false, EPI_GLU>,
        (const void*)gemm_kernel<true, EPI_BF16>,  (const void*)gemm_kernel<true, EPI_F32>,
        (const void*)gemm_kernel<true, EPI_RESID>,  (const void*)gemm_kernel<true, EPI_GLU>};
    for (const void* k : ks) {
      err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (err != cudaSuccess) break;
    }
  });
  if (err != cudaSuccess) return fail(SUB_ECUDA, std::string("gemm_init: ") + cudaGetErrorString(err));
  return SUB_OK;
}

template <bool W4, int EPI>
static int32_t gemm_launch(const GemvArgs& a, cudaStream_t st) {
  static_assert(BM * EPI_LD * 4 <= SMEM_BYTES, "epilogue tile must fit the pipeline buffers");
  SUB_TRY(gemm_init());
  auto kern = gemm_kernel<W4, EPI>;
  const int cols = (EPI == EPI_GLU) ? BN / 2 : BN;
  dim3 grid((a.N + cols - 1) / cols, (a.M + BM - 1) / BM);
  SUB_CUDA_TRY(launch_k(kern, grid, dim3(THREADS), SMEM_BYTES, st, a));
  return SUB_OK;
}

template <bool W4>
static int32_t gemm_epi(const GemvArgs& a, int epi, cudaStream_t st) {
  switch (epi) {
    case EPI_BF16: return gemm_launch<W4, EPI_BF16>(a, st);
    case EPI_F32: return gemm_launch<W4, EPI_F32>(a, st);
    case EPI_RESID: return gemm_launch<W4, EPI_RESID>(a, st);
    case EPI_GLU: return gemm_launch<W4, EPI_GLU>(a, st);
  }
  return fail(SUB_EINVAL, "bad gemm epilogue");
}

int32_t launch_gemm(const GemvArgs& a, bool is_w4, int epi, cudaStream_t st) {
  SUB_CHECK_ARG(a.M >= 1, "gemm: M must be positive");
  SUB_CHECK_ARG(a.K % 8 == 0 && a.ldx % 8 == 0, "gemm: K and ldx must be multiples of 8");
  SUB_CHECK_ARG(a.n_seg >= 1 && a.n_seg <= 4, "gemm: 1..4 segments");
  SUB_CHECK_ARG((int64_t)a.M < (1ll << 20), "gemm: M too large");
  SUB_CHECK_ARG(!a.xscale.partial && !(epi == EPI_RESID && a.norm.xn),
                "gemm: factored-norm inputs and outputs are GEMV-only");
  bool done = false;
  SUB_TRY(launch_gemm_tc(a, is_w4, epi, st, &done));
  if (done) return SUB_OK;
  return is_w4 ? gemm_epi<true>(a, epi, st) : gemm_epi<false>(a, epi, st);
}

}  // namespace sub
