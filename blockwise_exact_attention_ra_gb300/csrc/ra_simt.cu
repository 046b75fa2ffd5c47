// fp32 CUDA-core kernels (exact fp32 arithmetic) and the row/elementwise
// kernels shared by every path: state initialisation, the rescaled merge,
// the final normalisation, fp16 operand copies and the backward D = dO . O.
//
// The fp32 forward follows the ring loop of "Ring Attention: Train 1M Tokens
// on 8GB GPUs in 2026" ("Building Ring Attention in PyTorch: The 200-Line
// Version") with the rescaled (max, exp_sum, weighted_output) merge of its
// "Gotchas and Failure Modes" section: one warp per query row walks the
// key/value blocks of its host in ring order (i - s) mod P, 32 keys at a
// time, keeping (m, l, o) in registers.
#include <math.h>

#include "ra_device.cuh"

namespace ra {

namespace {

constexpr int kWarpsPerBlock = 4;

__device__ __forceinline__ void store_dtype(void* base, int dtype, long long idx,
                                            float x) {
  if (dtype == RA_F32)
    static_cast<float*>(base)[idx] = x;
  else if (dtype == RA_BF16)
    static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
  else
    static_cast<__half*>(base)[idx] = __float2half_rn(x);
}

__device__ __forceinline__ float load_dtype(const void* base, int dtype, long long idx) {
  if (dtype == RA_F32) return static_cast<const float*>(base)[idx];
  if (dtype == RA_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
  return __half2float(static_cast<const __half*>(base)[idx]);
}

__device__ __forceinline__ int clamp_len(const int* hl, int j, int S) {
  const int v = __ldg(hl + j);
  return v < 0 ? 0 : (v > S ? S : v);
}

// Keys [kbeg, kend) of one block against the warp's query row.  q_s holds the
// query row (d floats); lane owns output columns lane + 32*t.
template <int DPL>
__device__ __forceinline__ void simt_fwd_range(const float* __restrict__ q_s,
                                               const float* __restrict__ kbase,
                                               const float* __restrict__ vbase,
                                               long long row_stride, int kbeg, int kend,
                                               float scale, float& m, float& l,
                                               float (&o)[DPL]) {
  constexpr int D = DPL * 32;
  const int lane = threadIdx.x & 31;
  for (int c = kbeg; c < kend; c += 32) {
    const int j = c + lane;
    float s = -INFINITY;
    if (j < kend) {
      const float* kr = kbase + (long long)j * row_stride;
      float acc = 0.f;
#pragma unroll 8
      for (int t = 0; t < D; ++t) acc = fmaf(q_s[t], kr[t], acc);
      s = acc * scale;
    }
    const float cmax = warp_max(s);
    if (cmax == -INFINITY) continue;
    const float m_new = fmaxf(m, cmax);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float p = (s == -INFINITY) ? 0.f : expf(s - m_new);
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int t = 0; t < DPL; ++t) o[t] *= alpha;
    const int cnt = min(32, kend - c);
    for (int jj = 0; jj < cnt; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float* vr = vbase + (long long)(c + jj) * row_stride;
#pragma unroll
      for (int t = 0; t < DPL; ++t) o[t] = fmaf(pj, vr[lane + 32 * t], o[t]);
    }
    m = m_new;
  }
}

template <int DPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    simt_fwd_kernel(const SimtFwdArgs a) {
  constexpr int D = DPL * 32;
  __shared__ float q_sh[kWarpsPerBlock][D];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + w;  // (b, h, i)
  const long long total = (long long)a.B * a.Hq * a.Nq;
  if (row >= total) return;
  const int i = (int)(row % a.Nq);
  const int h = (int)((row / a.Nq) % a.Hq);
  const int b = (int)(row / ((long long)a.Nq * a.Hq));
  const int g = h / (a.Hq / a.Hkv);

  const float* qr = a.q + lay_at(a.ql, b, i, h);
#pragma unroll
  for (int t = 0; t < DPL; ++t) q_sh[w][lane + 32 * t] = qr[lane + 32 * t];
  __syncwarp();

  const long long kv_row_stride = a.kvl.rs;
  const float* kbase = a.k + lay_at(a.kvl, b, 0, g);
  const float* vbase = a.v + lay_at(a.kvl, b, 0, g);

  float m, l, o[DPL];
  const long long srow = ((long long)b * a.Hq + h) * a.Nq + i;       // m/l/lse index
  const long long orow = (((long long)b * a.Nq + i) * a.Hq + h) * D;  // packed o index
  if (a.P > 0) {
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) o[t] = 0.f;
    const int hi = i / a.S;
    const bool padded = a.host_len && (i - hi * a.S) >= clamp_len(a.host_len, hi, a.S);
    for (int s = 0; s < a.P; ++s) {
      const int blk = (hi - s + a.P) % a.P;
      const int kbeg = blk * a.S;
      int kend = kbeg + a.S;
      if (a.causal && a.striped) {
        // striped rows: local key row lk is visible iff lk < li, or lk == li
        // and the key's host is not after the query's
        kend = kbeg + (i - hi * a.S) + 1 - (blk > hi ? 1 : 0);
      } else if (a.causal) {
        if (blk > hi) continue;
        kend = min(kend, i + 1);
      }
      if (a.host_len) kend = min(kend, kbeg + clamp_len(a.host_len, blk, a.S));
      if (padded) break;  // padded query rows: O = 0, LSE = -inf
      simt_fwd_range<DPL>(q_sh[w], kbase, vbase, kv_row_stride, kbeg, kend, a.scale, m, l,
                          o);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const long long out_idx = lay_at(a.ql, b, i, h);
#pragma unroll
    for (int t = 0; t < DPL; ++t) store_dtype(a.o_out, a.o_dtype, out_idx + lane + 32 * t, o[t] * inv);
    if (lane == 0) a.lse[srow] = l > 0.f ? m + logf(l) : -INFINITY;
  } else {
    m = a.m_acc[srow];
    l = a.l_acc[srow];
#pragma unroll
    for (int t = 0; t < DPL; ++t) o[t] = a.o_acc[orow + lane + 32 * t];
    int kend = a.Nkv;
    if (a.causal) {
      const long long lim = a.q_off + i - a.kv_off + 1;  // keys with kv_pos <= q_pos
      kend = (int)max(0LL, min((long long)a.Nkv, lim));
    }
    simt_fwd_range<DPL>(q_sh[w], kbase, vbase, kv_row_stride, 0, kend, a.scale, m, l, o);
#pragma unroll
    for (int t = 0; t < DPL; ++t) a.o_acc[orow + lane + 32 * t] = o[t];
    if (lane == 0) {
      a.m_acc[srow] = m;
      a.l_acc[srow] = l;
    }
  }
}

// dQ rows: one warp per query row, keys in ring order.
template <int DPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) simt_bwd_dq_kernel(const SimtBwdArgs a) {
  constexpr int D = DPL * 32;
  __shared__ float q_sh[kWarpsPerBlock][D];
  __shared__ float do_sh[kWarpsPerBlock][D];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + w;
  if (row >= (long long)a.B * a.Hq * a.N) return;
  const int i = (int)(row % a.N);
  const int h = (int)((row / a.N) % a.Hq);
  const int b = (int)(row / ((long long)a.N * a.Hq));
  const int g = h / (a.Hq / a.Hkv);
  const long long qoff = lay_at(a.ql, b, i, h);
#pragma unroll
  for (int t = 0; t < DPL; ++t) {
    q_sh[w][lane + 32 * t] = a.q[qoff + lane + 32 * t];
    do_sh[w][lane + 32 * t] = a.dO[qoff + lane + 32 * t];
  }
  __syncwarp();
  const long long srow = ((long long)b * a.Hq + h) * a.N + i;
  const float lse = a.lse[srow];
  const float Di = a.Dvec[srow];
  const long long rs = a.kvl.rs;
  const float* kbase = a.k + lay_at(a.kvl, b, 0, g);
  const float* vbase = a.v + lay_at(a.kvl, b, 0, g);
  float dq[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) dq[t] = 0.f;
  const int hi = i / a.S;
  const bool padded = a.host_len && (i - hi * a.S) >= clamp_len(a.host_len, hi, a.S);
  for (int s = 0; s < a.P && !padded; ++s) {
    const int blk = (hi - s + a.P) % a.P;
    const int kbeg = blk * a.S;
    int kend = kbeg + a.S;
    if (a.causal && a.striped) {
      kend = kbeg + (i - hi * a.S) + 1 - (blk > hi ? 1 : 0);
    } else if (a.causal) {
      if (blk > hi) continue;
      kend = min(kend, i + 1);
    }
    if (a.host_len) kend = min(kend, kbeg + clamp_len(a.host_len, blk, a.S));
    for (int c = kbeg; c < kend; c += 32) {
      const int j = c + lane;
      float ds = 0.f;
      if (j < kend && lse != -INFINITY) {
        const float* kr = kbase + (long long)j * rs;
        const float* vr = vbase + (long long)j * rs;
        float sacc = 0.f, dpacc = 0.f;
#pragma unroll 8
        for (int t = 0; t < D; ++t) {
          sacc = fmaf(q_sh[w][t], kr[t], sacc);
          dpacc = fmaf(do_sh[w][t], vr[t], dpacc);
        }
        const float p = expf(sacc * a.scale - lse);
        ds = p * (dpacc - Di);
      }
      const int cnt = min(32, kend - c);
      for (int jj = 0; jj < cnt; ++jj) {
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
        const float* kr = kbase + (long long)(c + jj) * rs;
#pragma unroll
        for (int t = 0; t < DPL; ++t) dq[t] = fmaf(dsj, kr[lane + 32 * t], dq[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < DPL; ++t) store_dtype(a.dq, a.grad_dtype, qoff + lane + 32 * t, dq[t] * a.scale);
}

// dK, dV rows: one warp per key row; the key/value block visits the hosts
// (j + s) mod P in ring order and sums over the query heads of its group.
template <int DPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) simt_bwd_dkdv_kernel(const SimtBwdArgs a) {
  constexpr int D = DPL * 32;
  __shared__ float k_sh[kWarpsPerBlock][D];
  __shared__ float v_sh[kWarpsPerBlock][D];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const long long row = (long long)blockIdx.x * kWarpsPerBlock + w;
  if (row >= (long long)a.B * a.Hkv * a.N) return;
  const int j = (int)(row % a.N);
  const int g = (int)((row / a.N) % a.Hkv);
  const int b = (int)(row / ((long long)a.N * a.Hkv));
  const long long koff = lay_at(a.kvl, b, j, g);
#pragma unroll
  for (int t = 0; t < DPL; ++t) {
    k_sh[w][lane + 32 * t] = a.k[koff + lane + 32 * t];
    v_sh[w][lane + 32 * t] = a.v[koff + lane + 32 * t];
  }
  __syncwarp();
  const int group = a.Hq / a.Hkv;
  const long long qrs = a.ql.rs;
  float dk[DPL], dv[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) dk[t] = dv[t] = 0.f;
  const int hj = j / a.S;
  const bool padded = a.host_len && (j - hj * a.S) >= clamp_len(a.host_len, hj, a.S);
  for (int hh = 0; hh < group && !padded; ++hh) {
    const int h = g * group + hh;
    const float* qbase = a.q + lay_at(a.ql, b, 0, h);
    const float* dobase = a.dO + lay_at(a.ql, b, 0, h);
    const long long sbase = ((long long)b * a.Hq + h) * a.N;
    for (int s = 0; s < a.P; ++s) {
      const int host = (hj + s) % a.P;
      int qbeg = host * a.S;
      const int qend = qbeg + a.S;
      int qlim = qend;
      if (a.host_len) qlim = host * a.S + clamp_len(a.host_len, host, a.S);
      if (a.causal && a.striped) {
        // striped rows: local query row lq sees this key iff lq > lj, or
        // lq == lj and the key's host is not after the query's
        qbeg += (j - hj * a.S) + (hj > host ? 1 : 0);
      } else if (a.causal) {
        if (host < hj) continue;
        qbeg = max(qbeg, j);
      }
      for (int c = qbeg; c < qlim; c += 32) {
        const int i = c + lane;
        float p = 0.f, ds = 0.f;
        if (i < qlim) {
          const float lse = a.lse[sbase + i];
          if (lse != -INFINITY) {
            const float* qr = qbase + (long long)i * qrs;
            const float* dr = dobase + (long long)i * qrs;
            float sacc = 0.f, dpacc = 0.f;
#pragma unroll 8
            for (int t = 0; t < D; ++t) {
              sacc = fmaf(qr[t], k_sh[w][t], sacc);
              dpacc = fmaf(dr[t], v_sh[w][t], dpacc);
            }
            p = expf(sacc * a.scale - lse);
            ds = p * (dpacc - a.Dvec[sbase + i]);
          }
        }
        const int cnt = min(32, qlim - c);
        for (int ii = 0; ii < cnt; ++ii) {
          const float pi = __shfl_sync(0xffffffffu, p, ii);
          const float dsi = __shfl_sync(0xffffffffu, ds, ii);
          const float* qr = qbase + (long long)(c + ii) * qrs;
          const float* dr = dobase + (long long)(c + ii) * qrs;
#pragma unroll
          for (int t = 0; t < DPL; ++t) {
            dv[t] = fmaf(pi, dr[lane + 32 * t], dv[t]);
            dk[t] = fmaf(dsi, qr[lane + 32 * t], dk[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < DPL; ++t) {
    store_dtype(a.dk, a.grad_dtype, koff + lane + 32 * t, dk[t] * a.scale);
    store_dtype(a.dv, a.grad_dtype, koff + lane + 32 * t, dv[t]);
  }
}

// ---------------------------------------------------------------------------
// Row / elementwise kernels
// ---------------------------------------------------------------------------
__global__ void acc_init_kernel(float* o, float* m, float* l, long long rows,
                                long long oelems) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < oelems; t += stride) {
    o[t] = 0.f;
    if (t < rows) {
      m[t] = -INFINITY;
      l[t] = 0.f;
    }
  }
}

// One warp per (b, n, h) row: a <- merge(a, b).
__global__ void merge_kernel(float* oa, float* ma, float* la, const float* ob,
                             const float* mb, const float* lb, int B, int N, int H,
                             int d) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const int n = (int)((row / H) % N);
  const int b = (int)(row / ((long long)H * N));
  const long long sidx = ((long long)b * H + h) * N + n;
  const float m1 = ma[sidx], m2 = mb[sidx];
  const float m = fmaxf(m1, m2);
  float w1 = 0.f, w2 = 0.f;
  if (m != -INFINITY) {
    w1 = (m1 == -INFINITY) ? 0.f : expf(m1 - m);
    w2 = (m2 == -INFINITY) ? 0.f : expf(m2 - m);
  }
  float* orow = oa + row * d;
  const float* brow = ob + row * d;
  for (int c = lane; c < d; c += 32) orow[c] = w1 * orow[c] + w2 * brow[c];
  if (lane == 0) {
    la[sidx] = w1 * la[sidx] + w2 * lb[sidx];
    ma[sidx] = m;
  }
}

__global__ void finalize_kernel(const float* o, const float* m, const float* l, void* out,
                                int out_dtype, Lay out_l, float* lse, int B, int N,
                                int H, int d) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const int n = (int)((row / H) % N);
  const int b = (int)(row / ((long long)H * N));
  const long long sidx = ((long long)b * H + h) * N + n;
  const float lv = l[sidx];
  const float inv = lv > 0.f ? 1.f / lv : 0.f;
  const long long oidx = lay_at(out_l, b, n, h);
  for (int c = lane; c < d; c += 32) store_dtype(out, out_dtype, oidx + c, o[row * d + c] * inv);
  if (lane == 0 && lse) lse[sidx] = lv > 0.f ? m[sidx] + logf(lv) : -INFINITY;
}

// 8 elements per thread; d % 8 == 0 and rows aligned to 8 elements.  The
// destination is packed [B, N, H, d] (thread t writes elements 8t .. 8t+7).
// Packed sources (rows of H*d elements) take the flat index within a batch;
// other layouts decode (b, n, h) per vector.
template <typename T, bool PACKED>
__global__ void to_f16_kernel(const T* __restrict__ src, Lay src_l,
                              __half* __restrict__ dst, int B, int N, int H, int d, int* status) {
  const int vpr = d / 8;  // 8-element vectors per row
  const long long vpb = (long long)N * H * vpr;  // per batch
  const long long total = vpb * B;
  const long long stride = (long long)gridDim.x * blockDim.x;
  bool bad = false;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += stride) {
    const T* s;
    if (PACKED) {
      const long long b = t / vpb;
      s = src + b * src_l.bs + (t - b * vpb) * 8;
    } else {
      const long long row = t / vpr;  // packed (b, n, h) row
      const int h = (int)(row % H);
      const long long bn = row / H;
      s = src + lay_at(src_l, bn / N, bn % N, h) + (t - row * vpr) * 8;
    }
    __align__(16) __half outv[8];
    if constexpr (sizeof(T) == 2) {
      const uint4 raw = *reinterpret_cast<const uint4*>(s);
      const T* xs = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float f = to_f32(xs[u]);
        if (fabsf(f) > 65504.f && isfinite(f)) bad = true;
        outv[u] = __float2half_rn(f);
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float f = to_f32(s[u]);
        if (fabsf(f) > 65504.f && isfinite(f)) bad = true;
        outv[u] = __float2half_rn(f);
      }
    }
    *reinterpret_cast<uint4*>(dst + t * 8) = *reinterpret_cast<const uint4*>(outv);
  }
  if (bad) report(status, RA_ERR_RANGE);
}

__global__ void bwd_dot_kernel(const void* dO, int do_dtype, const void* o, int o_dtype,
                               Lay ql, float* D, const float* lse, float* lse2, int B,
                               int N, int H, int d) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const int n = (int)((row / H) % N);
  const int b = (int)(row / ((long long)H * N));
  const long long base = lay_at(ql, b, n, h);
  float acc = 0.f;
  for (int c = lane; c < d; c += 32)
    acc = fmaf(load_dtype(dO, do_dtype, base + c), load_dtype(o, o_dtype, base + c), acc);
  acc = warp_sum(acc);
  if (lane == 0) {
    const long long sidx = ((long long)b * H + h) * N + n;
    if (lse2) {  // tensor-core backward: -D and -LSE*log2(e), added with packed fp32 ops
      D[sidx] = -acc;
      lse2[sidx] = -(lse[sidx] * 1.4426950408889634f);
    } else {
      D[sidx] = acc;
    }
  }
}

// Packed destinations: one element per thread, flat index within a batch.
__global__ void f32_to_kernel(const float* __restrict__ src, void* out, int out_dtype,
                              long long out_bs, int B, long long epb, float mul) {
  const long long total = epb * B;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += stride) {
    const long long b = t / epb, e = t - b * epb;
    store_dtype(out, out_dtype, b * out_bs + e, src[t] * mul);
  }
}

// Other layouts: one warp per (b, n, h) row.
__global__ void f32_to_rows_kernel(const float* __restrict__ src, void* out, int out_dtype,
                                   Lay out_l, int B, int N, int H, int d, float mul) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * N * H) return;
  const int h = (int)(row % H);
  const long long bn = row / H;
  const long long o = lay_at(out_l, bn / N, bn % N, h);
  for (int c = lane; c < d; c += 32) store_dtype(out, out_dtype, o + c, src[row * d + c] * mul);
}

// One warp per (b, row): zero padded rows, set their LSE to -inf.
__global__ void fill_padding_kernel(void* t, int dtype, Lay l, int B, int N, int H, int d,
                                    int P, const int* host_len, float* lse) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * N) return;
  const int n = (int)(row % N), b = (int)(row / N);
  const int S = N / P;
  const int host = n / S;
  if (n - host * S < clamp_len(host_len, host, S)) return;
  for (int h = 0; h < H; ++h) {
    const long long base = lay_at(l, b, n, h);
    for (int c = lane; c < d; c += 32) store_dtype(t, dtype, base + c, 0.f);
  }
  if (lse)
    for (int h = lane; h < H; h += 32) lse[((long long)b * H + h) * N + n] = -INFINITY;
}

// One CTA waits on an mbarrier that nothing will ever arrive at; the bounded
// wait must give up, record RA_ERR_TIMEOUT and let the kernel return.
__global__ void selftest_timeout_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
  }
  __syncthreads();
}

unsigned grid_for(long long work, int per_block) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > (1LL << 30)) g = (1LL << 30);
  return (unsigned)g;
}

}  // namespace

cudaError_t launch_simt_fwd(const SimtFwdArgs& a, cudaStream_t st) {
  const long long rows = (long long)a.B * a.Hq * a.Nq;
  const unsigned grid = grid_for(rows, kWarpsPerBlock);
  const dim3 blk(kWarpsPerBlock * 32);
  switch (a.d) {
    case 32: simt_fwd_kernel<1><<<grid, blk, 0, st>>>(a); break;
    case 64: simt_fwd_kernel<2><<<grid, blk, 0, st>>>(a); break;
    case 128: simt_fwd_kernel<4><<<grid, blk, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd(const SimtBwdArgs& a, cudaStream_t st) {
  const unsigned gq = grid_for((long long)a.B * a.Hq * a.N, kWarpsPerBlock);
  const unsigned gk = grid_for((long long)a.B * a.Hkv * a.N, kWarpsPerBlock);
  const dim3 blk(kWarpsPerBlock * 32);
  switch (a.d) {
    case 32:
      simt_bwd_dq_kernel<1><<<gq, blk, 0, st>>>(a);
      simt_bwd_dkdv_kernel<1><<<gk, blk, 0, st>>>(a);
      break;
    case 64:
      simt_bwd_dq_kernel<2><<<gq, blk, 0, st>>>(a);
      simt_bwd_dkdv_kernel<2><<<gk, blk, 0, st>>>(a);
      break;
    case 128:
      simt_bwd_dq_kernel<4><<<gq, blk, 0, st>>>(a);
      simt_bwd_dkdv_kernel<4><<<gk, blk, 0, st>>>(a);
      break;
    default: return cudaErrorInvalidValue;
  }
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t launch_acc_init(float* o, float* m, float* l, int B, int N, int H, int d,
                            cudaStream_t st) {
  const long long rows = (long long)B * N * H;
  const long long oel = rows * d;
  acc_init_kernel<<<grid_for(oel, 256 * 8), 256, 0, st>>>(o, m, l, rows, oel);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge(float* oa, float* ma, float* la, const float* ob, const float* mb,
                         const float* lb, int B, int N, int H, int d, cudaStream_t st) {
  const long long rows = (long long)B * N * H;
  merge_kernel<<<grid_for(rows, 8), 256, 0, st>>>(oa, ma, la, ob, mb, lb, B, N, H, d);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* o, const float* m, const float* l, void* out,
                            int out_dtype, Lay out_l, float* lse, int B, int N, int H,
                            int d, cudaStream_t st) {
  const long long rows = (long long)B * N * H;
  finalize_kernel<<<grid_for(rows, 8), 256, 0, st>>>(o, m, l, out, out_dtype, out_l, lse, B,
                                                      N, H, d);
  count_launch();
  return cudaGetLastError();
}

template <typename T>
void to_f16_launch(const T* src, Lay src_l, __half* dst, int B, int N, int H, int d, int* status,
                   cudaStream_t st) {
  const unsigned grid = grid_for((long long)B * N * H * (d / 8), 256 * 4);
  if (src_l.rs == (long long)H * d && src_l.hs == d)
    to_f16_kernel<T, true><<<grid, 256, 0, st>>>(src, src_l, dst, B, N, H, d, status);
  else
    to_f16_kernel<T, false><<<grid, 256, 0, st>>>(src, src_l, dst, B, N, H, d, status);
}

cudaError_t launch_to_f16(const void* src, int src_dtype, Lay src_l, void* dst, int B, int N,
                          int H, int d, int* status, cudaStream_t st) {
  if (src_dtype == RA_BF16)
    to_f16_launch(static_cast<const __nv_bfloat16*>(src), src_l, static_cast<__half*>(dst), B, N, H, d,
                  status, st);
  else if (src_dtype == RA_F32)
    to_f16_launch(static_cast<const float*>(src), src_l, static_cast<__half*>(dst), B, N, H, d, status, st);
  else
    to_f16_launch(static_cast<const __half*>(src), src_l, static_cast<__half*>(dst), B, N, H, d, status, st);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_dot(const void* dO, int do_dtype, const void* o, int o_dtype,
                           Lay ql, float* D, const float* lse, float* lse2, int B,
                           int N, int H, int d, cudaStream_t st) {
  const long long rows = (long long)B * N * H;
  bwd_dot_kernel<<<grid_for(rows, 8), 256, 0, st>>>(dO, do_dtype, o, o_dtype, ql, D, lse,
                                                     lse2, B, N, H, d);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_f32_to(const float* src, void* out, int out_dtype, Lay out_l, int B, int N,
                          int H, int d, float mul, cudaStream_t st) {
  const long long epb = (long long)N * H * d;
  if (out_l.rs == (long long)H * d && out_l.hs == d)
    f32_to_kernel<<<grid_for(epb * B, 256 * 8), 256, 0, st>>>(src, out, out_dtype, out_l.bs, B, epb, mul);
  else
    f32_to_rows_kernel<<<grid_for((long long)B * N * H, 8), 256, 0, st>>>(src, out, out_dtype, out_l, B, N,
                                                                           H, d, mul);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_fill_padding(void* t, int dtype, Lay l, int B, int N, int H, int d, int P,
                                const int* host_len, float* lse, cudaStream_t st) {
  fill_padding_kernel<<<grid_for((long long)B * N, 8), 256, 0, st>>>(t, dtype, l, B, N, H, d, P, host_len,
                                                                      lse);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned int timeout_us, int* status, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>((unsigned long long)timeout_us * 1000ull, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace ra
