// Internal interface between the C-ABI front end (ra_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ra.h"

namespace ra {

// Division by a divisor that is fixed for a launch or a work unit, done as a
// multiply and a shift (the invariant-divisor method of Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", 1994):
// with m = floor(2^40 / d) + 1, floor(n * m / 2^40) = floor(n / d) for all
// 0 <= n < 2^20 and 1 <= d < 2^20, because the excess n * (m - 2^40 / d) / 2^40
// stays below 2^-20 < 1 / d.  Tile and iteration indices stay far below 2^20.
__host__ __device__ inline unsigned long long div_magic(unsigned d) { return (1ull << 40) / d + 1; }
__host__ __device__ inline int div_by(int n, unsigned long long m) {
  return (int)(((unsigned long long)(unsigned)n * m) >> 40);
}

// Layout of a [B, N, H, d] tensor with d contiguous: element (b, n, h, c)
// sits at b * bs + n * rs + h * hs + c (elements).  Packed: rs = H * d,
// hs = d, bs = N * H * d.
struct Lay {
  long long bs, rs, hs;
};
__host__ __device__ inline long long lay_at(const Lay& L, long long b, long long n, long long h) {
  return b * L.bs + n * L.rs + h * L.hs;
}
inline Lay packed_lay(long long N, long long H, long long d) { return Lay{N * H * d, H * d, d}; }

// ---------------------------------------------------------------------------
// fp32 CUDA-core path
// ---------------------------------------------------------------------------
struct SimtFwdArgs {
  const float* q;
  const float* k;
  const float* v;
  int B, Nq, Nkv, Hq, Hkv, d;
  Lay ql, kvl;              // q; k and v
  float scale;
  int causal;
  long long q_off, kv_off;  // block mode: global positions of row 0
  int P, S;                 // ring mode: P hosts of S rows; P == 0 -> block mode
  int striped;              // ring mode, causal: rows in striped order (position l*P + host)
  const int* host_len;      // ring mode, optional: valid rows per host (device, P entries)
  float* o_acc;             // block mode state (read + written)
  float* m_acc;
  float* l_acc;
  void* o_out;              // ring mode outputs (layout ql)
  int o_dtype;
  float* lse;
};

struct SimtBwdArgs {
  const float* q;
  const float* k;
  const float* v;
  const float* dO;
  const float* lse;
  const float* Dvec;  // [B, Hq, N]
  int B, N, Hq, Hkv, d;
  Lay ql, kvl;        // q, dO, dq; k, v, dk, dv
  float scale;
  int causal;
  int P, S;
  int striped;
  const int* host_len;
  void* dq;
  void* dk;
  void* dv;
  int grad_dtype;
};

cudaError_t launch_simt_fwd(const SimtFwdArgs& a, cudaStream_t st);
cudaError_t launch_simt_bwd(const SimtBwdArgs& a, cudaStream_t st);

// ---------------------------------------------------------------------------
// Elementwise / row kernels (any path)
// ---------------------------------------------------------------------------
cudaError_t launch_acc_init(float* o, float* m, float* l, int B, int N, int H, int d,
                            cudaStream_t st);
cudaError_t launch_merge(float* oa, float* ma, float* la, const float* ob,
                         const float* mb, const float* lb, int B, int N, int H, int d,
                         cudaStream_t st);
cudaError_t launch_finalize(const float* o, const float* m, const float* l, void* out,
                            int out_dtype, Lay out_l, float* lse, int B, int N,
                            int H, int d, cudaStream_t st);
// dst (packed fp16 [B, N, H, d]) <- src (dtype, layout src_l; rows 16-byte
// aligned, d % 8 == 0); values beyond the fp16 range set RA_ERR_RANGE in *status.
cudaError_t launch_to_f16(const void* src, int src_dtype, Lay src_l, void* dst,
                          int B, int N, int H, int d, int* status, cudaStream_t st);
// D[b, h, n] = sum_c dO[b, n, h, c] * O[b, n, h, c].  When lse2 is given (the
// tensor-core backward) both come out negated: D[b, h, n] = -sum(...) and
// lse2[b, h, n] = -lse[b, h, n] * log2(e), the terms that kernel adds.
cudaError_t launch_bwd_dot(const void* dO, int do_dtype, const void* o, int o_dtype,
                           Lay ql, float* D, const float* lse, float* lse2, int B,
                           int N, int H, int d, cudaStream_t st);
// out (dtype, layout out_l) <- mul * src (packed fp32 [B, N, H, d])
cudaError_t launch_f32_to(const float* src, void* out, int out_dtype, Lay out_l,
                          int B, int N, int H, int d, float mul, cudaStream_t st);
// Padded rows of a [B, N, H, d] tensor (row l of host i with l >= host_len[i],
// S = N / P rows per host) are set to zero, and lse[b, h, row] to -inf when
// lse is given.
cudaError_t launch_fill_padding(void* t, int dtype, Lay l, int B, int N, int H, int d,
                                int P, const int* host_len, float* lse, cudaStream_t st);
cudaError_t launch_selftest_timeout(unsigned int timeout_us, int* status,
                                    cudaStream_t st);

// Debug record of the tiles the tensor-core kernels bring in (see
// ra_debug_visit_log in ra.h): entries of four uint32, appended through an
// atomic cursor; entries past `capacity` are counted but not stored.
struct VisitLog {
  uint4* entries;
  unsigned int* count;
  unsigned long long capacity;
};

// ---------------------------------------------------------------------------
// tcgen05 tensor-core path (d = 64 or 128, fp16/bf16 operands)
// ---------------------------------------------------------------------------
struct TcFwdArgs {
  // Tensor maps over [B, N, H, d] (dims d, H, N, B), 64-element boxes of 128
  // rows, 128-byte swizzle.  q/k in qk_dtype, v in fp16.
  CUtensorMap tm_q, tm_k, tm_v;
  int qk_bf16;  // 1: q, k are bf16; 0: fp16
  int precise;  // two-term fp16 P in the P V product
  int B, Nq, Nkv, Hq, Hkv, d;
  float scale_log2;  // scale * log2(e)
  int causal;
  long long q_off, kv_off;
  int ring_P, ring_S;  // ring mode when ring_P > 0 (Nq == Nkv == P*S, S % 128 == 0)
  unsigned long long T_m;  // ring mode: div_magic(ring_S / 128)
  int striped;         // ring mode, causal: rows are in striped order (position l*P + host)
  const int* host_len; // ring mode, optional: valid rows per host (device, P entries)
  // outputs
  int mode;         // 0: ring (finalise), 1: block (read/write state)
  float* o_acc;     // block mode: [B, Nq, Hq, d] fp32
  float* m_acc;     // [B, Hq, Nq] (natural-log units)
  float* l_acc;
  void* o_out;      // ring mode: [B, Nq, Hq, d] in o_dtype, layout ol
  int o_dtype;
  Lay ol;
  float* lse;       // [B, Hq, Nq]
  int* status;
  unsigned long long wait_limit_ns;
  int num_units;    // work units (pairs of 128-row query tiles)
  unsigned int* sched;  // unit counter the CTAs draw from, zero at launch; NULL: CTA c takes units c, c + grid, ...
  VisitLog log;     // debug record of the key/value tiles loaded (off when log.entries is NULL)
};
cudaError_t launch_tc_fwd(TcFwdArgs& a, int num_sms, cudaStream_t st);

struct TcBwdArgs {
  // fp16 operands: q, dO over [B, N, Hq, d]; k, v over [B, N, Hkv, d]
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  // the fp32 dQ accumulator [B, N, Hq, d]: 32-column boxes of 128 rows,
  // 128-byte swizzle, written by TMA reduce-add
  CUtensorMap tm_dq;
  int B, N, Hq, Hkv, d;
  float scale;
  float scale_log2;
  int causal;
  int precise;  // two-term fp16 dS in the dK product
  int ring_P, ring_S;
  unsigned long long T_m;  // div_magic(ring_S / 128)
  unsigned long long P_m;  // div_magic(ring_P)
  int striped;  // causal, rows in striped order (position l*P + host)
  const int* host_len;  // optional: valid rows per host (device, P entries)
  const float* lse;   // [B, Hq, N]: -LSE * log2(e)
  const float* Dvec;  // [B, Hq, N]: -D
  float* dq_acc;      // packed fp32 [B, N, Hq, d], pre-zeroed, reduce-added
  void* dk;           // [B, N, Hkv, d] in grad_dtype, layout kvl
  void* dv;
  int grad_dtype;
  Lay kvl;
  int* status;
  unsigned long long wait_limit_ns;
  int num_units;
  unsigned int* sched;  // unit counter the CTAs draw from; zero at launch
  VisitLog log;     // debug record of the query tiles loaded (off when log.entries is NULL)
};
cudaError_t launch_tc_bwd(TcBwdArgs& a, int num_sms, cudaStream_t st);

// Counts kernel launches (ra_launch_count).
void count_launch(unsigned n = 1);

// Records `msg` as the calling thread's ra_last_error() message; returns code.
int set_error(int code, const char* msg);

// Row-major 16-bit matrix [rows, cols], leading dimension ld (elements):
// tensor map with box (64 columns, box_rows rows), 128-byte swizzle.
int make_map_2d(CUtensorMap* m, const void* base, int is_bf16, long long rows, long long cols,
                long long ld, int box_rows);

// ----------------------------------------------------------------- GEMM
// C[M, N] = epilogue(sum_k A(m, k) B(n, k)) on the tensor cores, 16-bit
// operands, fp32 accumulation.  A is K-major (a row-major [M, K] matrix) or
// MN-major (a row-major [K, M] matrix); B likewise with N.  Tiles 128 x 256.
enum GemmEpi {
  GEMM_STORE = 0,   // c = acc (c_dtype)
  GEMM_GELU = 1,    // c = GELU(acc) (16-bit)
  GEMM_GELU2 = 2,   // c = GELU(acc), c2 = GELU'(acc) (16-bit)
  GEMM_MUL = 3,     // c = acc * aux (16-bit aux and c)
  GEMM_ACC = 4,     // c += acc (fp32)
};
struct GemmArgs {
  CUtensorMap tm_a;   // K-major: box (64, 128); MN-major: box (64, 64)
  CUtensorMap tm_b;   // K-major: box (64, 256); MN-major: box (64, 64)
  int M, N, K;
  int a_mn, b_mn;
  int ab_bf16;        // operand type: bf16 (1) or fp16 (0)
  int epi;
  void* c;            // row-major [M, N], leading dimension ldc
  long long ldc;
  int c_dtype;        // ra_dtype of c
  void* c2;           // GEMM_GELU2: second output, same layout and type as c
  const void* aux;    // GEMM_MUL: row-major [M, N], leading dimension ldc, 16-bit
  // optional second problem of the same kind in the same launch (same K,
  // operand types and epilogue): its tiles follow the first problem's
  int groups;         // 1 or 2
  CUtensorMap tm_a2, tm_b2;
  int M2, N2;
  void* c_g2;
  long long ldc_g2;
  int* status;
  unsigned long long wait_limit_ns;
};
cudaError_t launch_tc_gemm(GemmArgs& a, int num_sms, cudaStream_t st);

}  // namespace ra
