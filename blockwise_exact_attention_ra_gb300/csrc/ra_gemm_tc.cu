// Tensor-core GEMM with fused epilogues, the building block of the blockwise
// feed-forward layer ("Ring Attention with Blockwise Transformers for
// Near-Infinite Context", Abstract: self-attention and the feedforward network
// are both computed blockwise).
//
// C[M, N] = epilogue(sum_k A(m, k) B(n, k)): 16-bit operands, fp32 accumulation
// in TMEM.  One persistent CTA per SM walks 128 x 256 output tiles:
//   warp 0      TMA producer: A and B k-slabs (64 deep) into a 4-stage ring,
//   warp 1      allocates TMEM, issues tcgen05.mma (M 128, N 256, K 16) into one
//               of two 256-column accumulators,
//   warps 2-9   epilogue: each reads 32 rows x 128 columns of the finished
//               accumulator, applies the epilogue and stores to global memory,
//               while the MMA warp fills the other accumulator.
// Operands are K-major (row-major [rows, K]: smem tile [rows][64] with the
// 128-byte swizzle) or MN-major (row-major [K, rows]: smem tile of 64-wide
// column chunks [chunk][64 k][64], chunk stride 8 KB).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ra_device.cuh"
#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kStageA = kBM * kBK * 2;          // 16 KB
constexpr int kStageB = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kStageA + kStageB;  // 48 KB
constexpr int kBars = kStages * kStageBytes;    // full[4], empty[4], acc_full[2], acc_empty[2], drain
constexpr int kMisc = kBars + 13 * 8;
constexpr int kUsed = kMisc + 16;
constexpr int kAlloc = kUsed + 1024;            // slack for 1024-byte alignment

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// GELU(u) = u Phi(u) and its derivative Phi(u) + u phi(u), with
// Phi(u) = (1 + erf(u / sqrt 2)) / 2 from Abramowitz and Stegun, Handbook of
// Mathematical Functions, formula 7.1.26: for x >= 0,
//   erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^{-x^2},
//   t = 1 / (1 + p x),  |error| <= 1.5e-7,
// whose e^{-x^2} = e^{-u^2/2} is also the exponential of phi(u).  One
// exponential and one reciprocal per element, against an erf and an exp;
// the error is far below the 16-bit rounding of the outputs.
template <bool GRAD>
__device__ __forceinline__ void gelu2_f(float2 u, float2* out, float2* grad) {
  // two elements at a time with the packed fp32x2 operations (FMA pipe)
  const float2 x = make_float2(fabsf(u.x) * 0.70710678118654752f, fabsf(u.y) * 0.70710678118654752f);
  const float2 d = __ffma2_rn(make_float2(0.3275911f, 0.3275911f), x, make_float2(1.f, 1.f));
  float2 t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t.x) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t.y) : "f"(d.y));
  const float2 uu = __fmul2_rn(u, u);
  // e^{-u^2/2} = 2^{-u^2 log2(e) / 2}
  const float2 e = make_float2(ex2_approx(-0.72134752044448170f * uu.x), ex2_approx(-0.72134752044448170f * uu.y));
  float2 p = __ffma2_rn(t, make_float2(1.061405429f, 1.061405429f), make_float2(-1.453152027f, -1.453152027f));
  p = __ffma2_rn(t, p, make_float2(1.421413741f, 1.421413741f));
  p = __ffma2_rn(t, p, make_float2(-0.284496736f, -0.284496736f));
  p = __ffma2_rn(t, p, make_float2(0.254829592f, 0.254829592f));
  p = __fmul2_rn(t, p);
  // (1 - poly e) / 2 = erf(|u| / sqrt 2) / 2
  const float2 h = __ffma2_rn(make_float2(-0.5f, -0.5f), __fmul2_rn(p, e), make_float2(0.5f, 0.5f));
  const float2 cdf = make_float2(0.5f + copysignf(h.x, u.x), 0.5f + copysignf(h.y, u.y));
  *out = __fmul2_rn(u, cdf);
  if (GRAD) *grad = __ffma2_rn(__fmul2_rn(u, make_float2(0.39894228040143268f, 0.39894228040143268f)), e, cdf);
}

__device__ __forceinline__ uint32_t pack16(float lo, float hi, int bf16) {
  if (bf16) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
  }
  __half2 t = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ float2 unpack16(uint32_t v, int bf16) {
  if (bf16) {
    __nv_bfloat162 t = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(t);
  }
  __half2 t = *reinterpret_cast<__half2*>(&v);
  return __half22float2(t);
}

// 32 consecutive 16-bit values of one row.
__device__ __forceinline__ void store16x32(void* p, const float* v, int bf16) {
  uint4* o = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    o[j] = make_uint4(pack16(v[8 * j], v[8 * j + 1], bf16), pack16(v[8 * j + 2], v[8 * j + 3], bf16),
                      pack16(v[8 * j + 4], v[8 * j + 5], bf16), pack16(v[8 * j + 6], v[8 * j + 7], bf16));
}

template <int A_MN, int B_MN, int EPI>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kBars;
  auto bar_full = [&](int s) { return bar0 + 8 * s; };
  auto bar_empty = [&](int s) { return bar0 + 8 * kStages + 8 * s; };
  auto bar_acc_full = [&](int b) { return bar0 + 16 * kStages + 8 * b; };
  auto bar_acc_empty = [&](int b) { return bar0 + 16 * kStages + 16 + 8 * b; };
  const uint32_t BAR_DRAIN = bar0 + 16 * kStages + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMisc + 4);
  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  // tiles of the first problem, then (grouped launch) of the second
  const int tiles_n = a.N / kBN;
  const int tiles0 = (a.M / kBM) * tiles_n;
  const int tiles_n2 = a.groups > 1 ? a.N2 / kBN : 1;
  const int num_tiles = tiles0 + (a.groups > 1 ? (a.M2 / kBM) * tiles_n2 : 0);
  const int k_steps = a.K / kBK;
  auto tile_at = [&](int t, int* m0, int* n0) {  // returns the problem index
    if (t < tiles0) {
      *m0 = (t / tiles_n) * kBM;
      *n0 = (t % tiles_n) * kBN;
      return 0;
    }
    t -= tiles0;
    *m0 = (t / tiles_n2) * kBM;
    *n0 = (t % tiles_n2) * kBN;
    return 1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full(b), 1);
      mbar_init(bar_acc_empty(b), kEpiWarps * 32);
    }
    mbar_init(BAR_DRAIN, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_b);
    if (a.groups > 1) {
      tma_prefetch_desc(&a.tm_a2);
      tma_prefetch_desc(&a.tm_b2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t lim = a.wait_limit_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      uint32_t cnt = 0;
      bool ok = true;
      int issued[kStages] = {0, 0, 0, 0};
      uint32_t last_phase[kStages] = {0, 0, 0, 0};
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int m0, n0;
        const int grp = tile_at(t, &m0, &n0);
        const CUtensorMap* ma = grp ? &a.tm_a2 : &a.tm_a;
        const CUtensorMap* mb = grp ? &a.tm_b2 : &a.tm_b;
        for (int kb = 0; kb < k_steps; ++kb, ++cnt) {
          const int s = cnt % kStages;
          const uint32_t ph = (cnt / kStages) & 1;
          if (!mbar_wait(bar_empty(s), ph ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_full(s), kStageBytes);
          const uint32_t dA = sbase + s * kStageBytes, dB = dA + kStageA;
          const int k0 = kb * kBK;
          if (A_MN) {
#pragma unroll
            for (int c = 0; c < kBM / 64; ++c) tma_load_2d(dA + c * 8192, ma, bar_full(s), m0 + 64 * c, k0, pol);
          } else {
            tma_load_2d(dA, ma, bar_full(s), k0, m0, pol);
          }
          if (B_MN) {
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c) tma_load_2d(dB + c * 8192, mb, bar_full(s), n0 + 64 * c, k0, pol);
          } else {
            tma_load_2d(dB, mb, bar_full(s), k0, n0, pol);
          }
          issued[s] = 1;
          last_phase[s] = ph;
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) (void)mbar_wait(bar_full(s), last_phase[s], abort_flag, nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(a.ab_bf16 ? 1u : 0u, A_MN, B_MN, kBM, kBN);
      // K-major: LBO unused, SBO = 8 rows x 128 B; MN-major: LBO = the 8 KB
      // chunk stride, SBO = 8 k-rows x 128 B.  One K = 16 step moves 32 B
      // (K-major) or 16 k-rows = 2 KB (MN-major).
      const uint64_t dA0 = smem_desc_sw128(sbase, A_MN ? 8192 : 16, 1024);
      const uint64_t dB0 = smem_desc_sw128(sbase + kStageA, B_MN ? 8192 : 16, 1024);
      constexpr uint32_t kStep = kStageBytes >> 4;
      constexpr uint32_t offA = A_MN ? 2048 : 32, offB = B_MN ? 2048 : 32;
      uint32_t cnt = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++lt) {
        const uint32_t b = lt & 1;
        if (!mbar_wait(bar_acc_empty(b), ((lt >> 1) & 1) ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + b * kBN;
        for (int kb = 0; kb < k_steps; ++kb, ++cnt) {
          const int s = cnt % kStages;
          if (!mbar_wait(bar_full(s), (cnt / kStages) & 1, abort_flag, a.status, lim)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = dA0 + s * kStep, db = dB0 + s * kStep;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_ss(acc, desc_off(da, kk * offA), desc_off(db, kk * offB), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar_empty(s));
        }
        if (!ok) break;
        mma_commit(bar_acc_full(b));
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(BAR_DRAIN);
      (void)mbar_wait(BAR_DRAIN, 0, abort_flag, nullptr, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
    const int half = (int)(warp - 2) >> 2;        // columns [128*half, 128*half + 128)
    const int bf16 = a.ab_bf16;
    uint32_t lt = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++lt) {
      const uint32_t b = lt & 1;
      if (!mbar_wait(bar_acc_full(b), (lt >> 1) & 1, abort_flag, a.status, lim)) { ok = false; break; }
      tc_fence_after();
      int m0, n0;
      const int grp = tile_at(t, &m0, &n0);
      void* cbase = grp ? a.c_g2 : a.c;
      const long long ldc = grp ? a.ldc_g2 : a.ldc;
      const long long row = (long long)m0 + quarter * 32 + lane;
      const int col0 = n0 + half * 128;
      const uint32_t src = tmem + b * kBN + half * 128 + ((quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < 128; c += 32) {
        uint32_t r[32];
        RA_TMEM_LD32(src + c, r);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        const long long off = row * ldc + col0 + c;
        if (EPI == GEMM_STORE) {
          if (a.c_dtype == RA_F32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(cbase) + off);
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            store16x32(static_cast<uint16_t*>(cbase) + off, v, a.c_dtype == RA_BF16);
          }
        } else if (EPI == GEMM_GELU) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float2 o;
            gelu2_f<false>(make_float2(v[j], v[j + 1]), &o, nullptr);
            v[j] = o.x;
            v[j + 1] = o.y;
          }
          store16x32(static_cast<uint16_t*>(cbase) + off, v, bf16);
        } else if (EPI == GEMM_GELU2) {
          float g[32];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float2 o, gr;
            gelu2_f<true>(make_float2(v[j], v[j + 1]), &o, &gr);
            v[j] = o.x;
            v[j + 1] = o.y;
            g[j] = gr.x;
            g[j + 1] = gr.y;
          }
          store16x32(static_cast<uint16_t*>(cbase) + off, v, bf16);
          store16x32(static_cast<uint16_t*>(a.c2) + off, g, bf16);
        } else if (EPI == GEMM_MUL) {
          const uint4* m = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.aux) + off);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = m[j];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = unpack16(ww[q], bf16);
              v[8 * j + 2 * q] *= f.x;
              v[8 * j + 2 * q + 1] *= f.y;
            }
          }
          store16x32(static_cast<uint16_t*>(cbase) + off, v, bf16);
        } else {  // GEMM_ACC
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(cbase) + off);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 x = o[j];
            x.x += v[4 * j];
            x.y += v[4 * j + 1];
            x.z += v[4 * j + 2];
            x.w += v[4 * j + 3];
            o[j] = x;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acc_empty(b));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tc_gemm(GemmArgs& a, int num_sms, cudaStream_t st) {
  if (a.M % kBM || a.N % kBN || a.K % kBK || a.M <= 0 || a.N <= 0 || a.K <= 0) return cudaErrorInvalidValue;
  if (a.groups < 1) a.groups = 1;
  if (a.groups > 2 || (a.groups == 2 && (a.M2 % kBM || a.N2 % kBN || a.M2 <= 0 || a.N2 <= 0)))
    return cudaErrorInvalidValue;
  const int tiles = (a.M / kBM) * (a.N / kBN) + (a.groups == 2 ? (a.M2 / kBM) * (a.N2 / kBN) : 0);
  const int grid = tiles < num_sms ? tiles : num_sms;
  auto run = [&](auto kernel) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, kAlloc, st>>>(a);
    return cudaSuccess;
  };
  cudaError_t e;
  if (!a.a_mn && !a.b_mn && a.epi == GEMM_STORE) e = run(tc_gemm_kernel<0, 0, GEMM_STORE>);
  else if (!a.a_mn && !a.b_mn && a.epi == GEMM_GELU) e = run(tc_gemm_kernel<0, 0, GEMM_GELU>);
  else if (!a.a_mn && !a.b_mn && a.epi == GEMM_GELU2) e = run(tc_gemm_kernel<0, 0, GEMM_GELU2>);
  else if (!a.a_mn && a.b_mn && a.epi == GEMM_MUL) e = run(tc_gemm_kernel<0, 1, GEMM_MUL>);
  else if (!a.a_mn && a.b_mn && a.epi == GEMM_STORE) e = run(tc_gemm_kernel<0, 1, GEMM_STORE>);
  else if (a.a_mn && a.b_mn && a.epi == GEMM_ACC) e = run(tc_gemm_kernel<1, 1, GEMM_ACC>);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace ra
