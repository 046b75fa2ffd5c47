// C-ABI front end of libra: argument validation, workspace layout, tensor
// map encoding and kernel dispatch.  Every entry point only enqueues work on
// the caller's stream; nothing here allocates device memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "ra_internal.h"

// One status word per device (module-global storage, not an allocation).
__device__ int g_ra_status_word;

namespace ra {

static std::atomic<unsigned long long> g_launches{0};
void count_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {

thread_local std::string t_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceCache {
  std::mutex mu;
  int* status[kMaxDevices] = {};
  int sms[kMaxDevices] = {};
  int cc_major[kMaxDevices] = {};
  int cc_minor[kMaxDevices] = {};
};
DeviceCache& cache() {
  static DeviceCache c;
  return c;
}

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device ordinal %d", *dev);
  return RA_OK;
}

// Address of this device's status word, looked up once per device.
int status_ptr(int** out) {
  int dev;
  int rc = current_device(&dev);
  if (rc) return rc;
  DeviceCache& c = cache();
  std::lock_guard<std::mutex> lk(c.mu);
  if (!c.status[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_ra_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    c.status[dev] = static_cast<int*>(p);
    cudaDeviceGetAttribute(&c.sms[dev], cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&c.cc_major[dev], cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&c.cc_minor[dev], cudaDevAttrComputeCapabilityMinor, dev);
  }
  *out = c.status[dev];
  return RA_OK;
}

int device_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  return cache().sms[dev] > 0 ? cache().sms[dev] : 1;
}

bool device_is_sm103() {
  int dev = 0;
  cudaGetDevice(&dev);
  return cache().cc_major[dev] == 10 && cache().cc_minor[dev] == 3;
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* s = getenv("RA_WAIT_TIMEOUT_MS");
    unsigned long long ms = s ? strtoull(s, nullptr, 10) : 10000ull;
    if (ms == 0) ms = 10000ull;
    return ms * 1000000ull;
  }();
  return v;
}

// -------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

int encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn f = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                           &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) f = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!f) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *fn = f;
  return RA_OK;
}

// [B, N, H, d] 16-bit tensor with layout L (elements): dims (d, H, N, B),
// box (64, 1, 128, 1), 128-byte swizzle; rows past N read as zeros.
int make_map(CUtensorMap* m, const void* base, int is_bf16, int B, int N, int H, int d,
             const Lay& L) {
  EncodeTiledFn fn;
  int rc = encoder(&fn);
  if (rc) return rc;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)L.hs * 2, (cuuint64_t)L.rs * 2, (cuuint64_t)L.bs * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return RA_OK;
}

// Packed fp32 [B, N, H, d] tensor: box (32, 1, 32, 1), 128-byte swizzle (one
// warp's 32 rows of a 32-column slab).
int make_map_f32(CUtensorMap* m, void* base, int B, int N, int H, int d) {
  EncodeTiledFn fn;
  int rc = encoder(&fn);
  if (rc) return rc;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4, (cuuint64_t)N * H * d * 4};
  cuuint32_t box[4] = {32, 1, 32, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled (fp32) failed (%d)", (int)r);
  return RA_OK;
}

}  // namespace

// Row-major 16-bit matrix [rows, cols] with leading dimension ld (elements):
// dims (cols, rows), box (64, box_rows), 128-byte swizzle.
int make_map_2d(CUtensorMap* m, const void* base, int is_bf16, long long rows, long long cols,
                long long ld, int box_rows) {
  EncodeTiledFn fn;
  int rc = encoder(&fn);
  if (rc) return rc;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled (2-D) failed (%d)", (int)r);
  return RA_OK;
}

namespace {

// -------------------------------------------------------------- validation
size_t dtype_size(int dt) { return dt == RA_F32 ? 4 : 2; }
bool valid_dtype(int dt) { return dt == RA_F32 || dt == RA_BF16 || dt == RA_F16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Shape {
  int B, Nq, Nkv, Hq, Hkv, d;
  Lay ql, kvl;  // q, o, dO, dq; k, v, dk, dv
};

// The layout of one group: zero strides take their packed defaults; rows of
// d elements at n * rs + h * hs must not overlap (the smaller of the two
// strides steps past a row, the larger past the whole inner axis), nor may
// one batch overlap the next.
int group_layout(const char* name, int N, int H, int d, long long bs, long long rs, long long hs, Lay* out) {
  if (bs < 0 || rs < 0 || hs < 0) return fail(RA_ERR_INVALID_ARG, "%s strides must be >= 0", name);
  if (rs == 0) rs = (long long)H * d;
  if (hs == 0) hs = d;
  long long s1 = rs, n1 = N, s2 = hs, n2 = H;
  if (s1 > s2) {
    long long t = s1; s1 = s2; s2 = t;
    t = n1; n1 = n2; n2 = t;
  }
  const long long inner = (n1 - 1) * s1 + d;
  if ((n1 > 1 && s1 < d) || (n2 > 1 && s2 < inner))
    return fail(RA_ERR_INVALID_ARG, "%s row and head strides (%lld, %lld) make rows of %d elements overlap", name,
                rs, hs, d);
  const long long extent = (long long)(N - 1) * rs + (long long)(H - 1) * hs + d;
  if (bs == 0) bs = extent;
  if (bs < extent)
    return fail(RA_ERR_INVALID_ARG, "%s batch stride %lld is smaller than one batch (%lld elements)", name, bs,
                extent);
  *out = Lay{bs, rs, hs};
  return RA_OK;
}

int check_shape(const ra_shape& s, Shape* out) {
  if (s.B < 1 || s.N_q < 1 || s.N_kv < 1 || s.Hq < 1 || s.Hkv < 1 || s.d < 1)
    return fail(RA_ERR_INVALID_ARG, "shape has a non-positive extent (B=%d N_q=%d N_kv=%d Hq=%d Hkv=%d d=%d)",
                s.B, s.N_q, s.N_kv, s.Hq, s.Hkv, s.d);
  if (s.Hq % s.Hkv) return fail(RA_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", s.Hq, s.Hkv);
  if (s.N_q >= (1 << 30) || s.N_kv >= (1 << 30) || s.Hq > 4096 || s.d > 4096)
    return fail(RA_ERR_INVALID_ARG, "shape extent too large");
  const long long big = 1ll << 50;  // keeps every offset product far from overflow
  if (s.q_bstride > big || s.kv_bstride > big || s.q_rstride > big || s.q_hstride > big || s.kv_rstride > big ||
      s.kv_hstride > big)
    return fail(RA_ERR_INVALID_ARG, "stride too large");
  Shape r{s.B, s.N_q, s.N_kv, s.Hq, s.Hkv, s.d, {}, {}};
  int rc;
  if ((rc = group_layout("q", s.N_q, s.Hq, s.d, s.q_bstride, s.q_rstride, s.q_hstride, &r.ql)) ||
      (rc = group_layout("kv", s.N_kv, s.Hkv, s.d, s.kv_bstride, s.kv_rstride, s.kv_hstride, &r.kvl)))
    return rc;
  *out = r;
  return RA_OK;
}

bool is_packed(const Lay& L, long long N, long long H, long long d) {
  return L.rs == H * d && L.hs == d;
}

int check_ptr(const void* p, const char* name) {
  if (!p) return fail(RA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(RA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return RA_OK;
}

int check_scale(float scale) {
  if (!(scale > 0.f) || !isfinite(scale))
    return fail(RA_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", (double)scale);
  return RA_OK;
}

// Tensor-core path prerequisites (d, strides, device).
int check_tc(const Shape& s, int dtype) {
  if (s.d != 64 && s.d != 128)
    return fail(RA_ERR_UNSUPPORTED, "tensor-core path supports d in {64, 128} (got %d)", s.d);
  for (const Lay* L : {&s.ql, &s.kvl})
    if ((L->bs % 8) || (L->rs % 8) || (L->hs % 8))
      return fail(RA_ERR_INVALID_ARG, "16-bit tensor-core inputs need strides that are multiples of 8 elements");
  if (!device_is_sm103())
    return fail(RA_ERR_UNSUPPORTED, "tensor-core kernels are built for sm_103a only");
  (void)dtype;
  return RA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------------------ kernel timing
struct KernelTimer {
  std::mutex mu;
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev[RA_KERNEL_COUNT];
};
KernelTimer& ktimer() {
  static KernelTimer t;
  return t;
}
void ktimer_clear(KernelTimer& t) {
  for (auto& v : t.ev) {
    for (auto& p : v) {
      cudaEventDestroy(p.first);
      cudaEventDestroy(p.second);
    }
    v.clear();
  }
}

// Brackets one launch with events when timing is on.
struct TimedLaunch {
  int id;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  TimedLaunch(int kid, cudaStream_t s) : id(kid), st(s) {
    KernelTimer& t = ktimer();
    std::lock_guard<std::mutex> lk(t.mu);
    if (!t.on) return;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
      a = b = nullptr;
      return;
    }
    cudaEventRecord(a, st);
  }
  ~TimedLaunch() {
    if (!a) return;
    cudaEventRecord(b, st);
    KernelTimer& t = ktimer();
    std::lock_guard<std::mutex> lk(t.mu);
    t.ev[id].emplace_back(a, b);
  }
};

}  // namespace

int set_error(int code, const char* msg) {
  t_err = msg;
  return code;
}

namespace {
// The debug visit log set by ra_debug_visit_log (process-wide; off by default).
std::mutex g_log_mu;
VisitLog g_log{nullptr, nullptr, 0};
VisitLog visit_log() {
  std::lock_guard<std::mutex> lk(g_log_mu);
  return g_log;
}
}  // namespace

}  // namespace ra

using namespace ra;

extern "C" {
#pragma GCC visibility push(default)

const char* ra_last_error(void) { return t_err.c_str(); }

unsigned long long ra_launch_count(void) { return g_launches.load(); }

int ra_debug_visit_log(unsigned int* entries, size_t capacity, unsigned int* count) {
  if (entries && (!count || capacity == 0))
    return fail(RA_ERR_INVALID_ARG, "a visit log needs a count word and a capacity > 0");
  if (entries && ((reinterpret_cast<uintptr_t>(entries) & 15u) || (reinterpret_cast<uintptr_t>(count) & 3u)))
    return fail(RA_ERR_INVALID_ARG, "visit log entries must be 16-byte aligned and the count word 4-byte aligned");
  std::lock_guard<std::mutex> lk(g_log_mu);
  if (entries)
    g_log = VisitLog{reinterpret_cast<uint4*>(entries), count, (unsigned long long)capacity};
  else
    g_log = VisitLog{nullptr, nullptr, 0};
  return RA_OK;
}

int ra_kernel_timing(int enable) {
  KernelTimer& t = ktimer();
  std::lock_guard<std::mutex> lk(t.mu);
  ktimer_clear(t);
  t.on = enable != 0;
  return RA_OK;
}

int ra_kernel_timing_read(int kernel, double* total_ms, unsigned long long* launches) {
  if (kernel < 0 || kernel >= RA_KERNEL_COUNT || !total_ms || !launches)
    return fail(RA_ERR_INVALID_ARG, "bad kernel id or NULL output");
  KernelTimer& t = ktimer();
  std::lock_guard<std::mutex> lk(t.mu);
  double sum = 0.0;
  for (auto& p : t.ev[kernel]) {
    cudaError_t e = cudaEventSynchronize(p.second);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, p.first, p.second);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    sum += ms;
  }
  *total_ms = sum;
  *launches = t.ev[kernel].size();
  return RA_OK;
}

int ra_sync_status(void* stream) {
  int* st;
  int rc = status_ptr(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_ra_status_word, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (v) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_ra_status_word, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    return fail(v, v == RA_ERR_RANGE ? "an operand exceeded the fp16 range"
                                     : v == RA_ERR_TIMEOUT ? "a bounded wait on the device gave up"
                                                           : "device reported status %d",
                v);
  }
  t_err.clear();
  return RA_OK;
}

int ra_selftest_timeout(unsigned int timeout_us, void* stream) {
  int* st;
  int rc = status_ptr(&st);
  if (rc) return rc;
  if (timeout_us == 0 || timeout_us > 10000000u)
    return fail(RA_ERR_INVALID_ARG, "timeout_us must be in (0, 1e7]");
  cudaError_t e = launch_selftest_timeout(timeout_us, st, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "selftest_timeout launch");
}

int ra_acc_init(float* o_acc, float* m_acc, float* l_acc, ra_shape shape, void* stream) {
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if ((rc = check_ptr(o_acc, "o_acc")) || (rc = check_ptr(m_acc, "m_acc")) || (rc = check_ptr(l_acc, "l_acc")))
    return rc;
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  cudaError_t e = launch_acc_init(o_acc, m_acc, l_acc, s.B, s.Nq, s.Hq, s.d,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "acc_init launch");
}

int ra_merge(float* o_a, float* m_a, float* l_a, const float* o_b, const float* m_b,
             const float* l_b, ra_shape shape, void* stream) {
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if ((rc = check_ptr(o_a, "o_a")) || (rc = check_ptr(m_a, "m_a")) || (rc = check_ptr(l_a, "l_a")) ||
      (rc = check_ptr(o_b, "o_b")) || (rc = check_ptr(m_b, "m_b")) || (rc = check_ptr(l_b, "l_b")))
    return rc;
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  cudaError_t e = launch_merge(o_a, m_a, l_a, o_b, m_b, l_b, s.B, s.Nq, s.Hq, s.d,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "merge launch");
}

int ra_finalize(const float* o_acc, const float* m_acc, const float* l_acc, void* o_out,
                ra_dtype o_dtype, float* lse, ra_shape shape, void* stream) {
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if (!valid_dtype(o_dtype)) return fail(RA_ERR_INVALID_ARG, "bad o_dtype %d", (int)o_dtype);
  if ((rc = check_ptr(o_acc, "o_acc")) || (rc = check_ptr(m_acc, "m_acc")) || (rc = check_ptr(l_acc, "l_acc")) ||
      (rc = check_ptr(o_out, "o_out")) || (rc = check_ptr(lse, "lse")))
    return rc;
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  cudaError_t e = launch_finalize(o_acc, m_acc, l_acc, o_out, o_dtype, s.ql, lse, s.B, s.Nq,
                                  s.Hq, s.d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "finalize launch");
}

size_t ra_block_fwd_workspace_bytes(ra_dtype dtype, ra_shape shape) {
  if (dtype != RA_BF16 || shape.B < 1 || shape.N_kv < 1 || shape.Hkv < 1 || shape.d < 1) return 0;
  return align256((size_t)shape.B * shape.N_kv * shape.Hkv * shape.d * 2);
}

int ra_block_fwd(const void* q, const void* k_blk, const void* v_blk, ra_dtype dtype,
                 float* o_acc, float* m_acc, float* l_acc, ra_shape shape, long long q_off,
                 long long kv_off, int flags, float scale, void* workspace, size_t ws_bytes,
                 void* stream) {
  const int causal = (flags & RA_CAUSAL) != 0, precise = (flags & RA_PRECISE) != 0;
  if (flags & ~(RA_CAUSAL | RA_PRECISE)) return fail(RA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if (!valid_dtype(dtype)) return fail(RA_ERR_INVALID_ARG, "bad dtype %d", (int)dtype);
  if ((rc = check_scale(scale))) return rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k_blk, "k_blk")) || (rc = check_ptr(v_blk, "v_blk")) ||
      (rc = check_ptr(o_acc, "o_acc")) || (rc = check_ptr(m_acc, "m_acc")) || (rc = check_ptr(l_acc, "l_acc")))
    return rc;
  if (q_off < 0 || kv_off < 0) return fail(RA_ERR_INVALID_ARG, "offsets must be >= 0");
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (dtype == RA_F32) {
    if (s.d != 32 && s.d != 64 && s.d != 128)
      return fail(RA_ERR_UNSUPPORTED, "fp32 path supports d in {32, 64, 128} (got %d)", s.d);
    SimtFwdArgs a{};
    a.q = static_cast<const float*>(q);
    a.k = static_cast<const float*>(k_blk);
    a.v = static_cast<const float*>(v_blk);
    a.B = s.B; a.Nq = s.Nq; a.Nkv = s.Nkv; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d;
    a.ql = s.ql; a.kvl = s.kvl;
    a.scale = scale; a.causal = causal; a.q_off = q_off; a.kv_off = kv_off;
    a.P = 0; a.S = 0;
    a.o_acc = o_acc; a.m_acc = m_acc; a.l_acc = l_acc;
    TimedLaunch tl(RA_KERNEL_FWD_F32, cs);
    cudaError_t e = launch_simt_fwd(a, cs);
    return e == cudaSuccess ? RA_OK : cuda_fail(e, "fp32 block forward launch");
  }
  if ((rc = check_tc(s, dtype))) return rc;
  const void* v16 = v_blk;
  if (dtype == RA_BF16) {
    const size_t need = ra_block_fwd_workspace_bytes(dtype, shape);
    if (!workspace || ws_bytes < need)
      return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
    if ((rc = check_ptr(workspace, "workspace"))) return rc;
    cudaError_t e = launch_to_f16(v_blk, RA_BF16, s.kvl, workspace, s.B, s.Nkv, s.Hkv, s.d, st, cs);
    if (e != cudaSuccess) return cuda_fail(e, "v -> fp16 launch");
    v16 = workspace;
  }
  TcFwdArgs a;
  memset(&a, 0, sizeof a);
  const int bf = dtype == RA_BF16;
  if ((rc = make_map(&a.tm_q, q, bf, s.B, s.Nq, s.Hq, s.d, s.ql))) return rc;
  if ((rc = make_map(&a.tm_k, k_blk, bf, s.B, s.Nkv, s.Hkv, s.d, s.kvl))) return rc;
  if ((rc = make_map(&a.tm_v, v16, 0, s.B, s.Nkv, s.Hkv, s.d,
                     dtype == RA_BF16 ? packed_lay(s.Nkv, s.Hkv, s.d) : s.kvl)))
    return rc;
  a.qk_bf16 = bf;
  a.B = s.B; a.Nq = s.Nq; a.Nkv = s.Nkv; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal; a.q_off = q_off; a.kv_off = kv_off; a.precise = precise;
  a.ring_P = 0; a.ring_S = 0; a.T_m = 0; a.mode = 1;
  a.o_acc = o_acc; a.m_acc = m_acc; a.l_acc = l_acc;
  a.status = st;
  a.wait_limit_ns = wait_limit_ns();
  a.log = visit_log();
  const int nqt = (s.Nq + 127) / 128;
  a.num_units = s.B * s.Hq * ((nqt + 1) / 2);
  TimedLaunch tl(RA_KERNEL_FWD_TC, cs);
  cudaError_t e = launch_tc_fwd(a, device_sms(), cs);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "tensor-core block forward launch");
}

// Ring forward workspace (16-bit dtypes): unit counter (256 bytes) | fp16
// copy of V [B,N,Hkv,d] (bf16 inputs).
size_t ra_ring_fwd_workspace_bytes(ra_dtype dtype, ra_shape shape, int P) {
  (void)P;
  if ((dtype != RA_BF16 && dtype != RA_F16) || shape.B < 1 || shape.N_kv < 1 || shape.Hkv < 1 || shape.d < 1)
    return 0;
  if (dtype == RA_F16) return 256;
  return 256 + align256((size_t)shape.B * shape.N_kv * shape.Hkv * shape.d * 2);
}

static int check_ring(const Shape& s, int P, int dtype) {
  if (s.Nq != s.Nkv) return fail(RA_ERR_INVALID_ARG, "ring attention needs N_q == N_kv (%d vs %d)", s.Nq, s.Nkv);
  if (P < 1 || s.Nq % P) return fail(RA_ERR_INVALID_ARG, "P=%d must divide N=%d", P, s.Nq);
  if (dtype != RA_F32 && (s.Nq / P) % 128)
    return fail(RA_ERR_UNSUPPORTED, "tensor-core ring needs a host block N/P that is a multiple of 128 (got %d)",
                s.Nq / P);
  return RA_OK;
}

static int ring_fwd_impl(const void* q, const void* k, const void* v, ra_dtype dtype, ra_shape shape,
                         int P, int flags, float scale, void* o, ra_dtype o_dtype, float* lse,
                         void* workspace, size_t ws_bytes, void* stream, const int* host_len) {
  const int causal = (flags & RA_CAUSAL) != 0, precise = (flags & RA_PRECISE) != 0;
  const int striped = causal && (flags & RA_STRIPED) != 0;
  if (flags & ~(RA_CAUSAL | RA_PRECISE | RA_STRIPED))
    return fail(RA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  if (host_len && striped)
    return fail(RA_ERR_INVALID_ARG, "RA_STRIPED does not combine with per-host lengths");
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if (!valid_dtype(dtype) || !valid_dtype(o_dtype)) return fail(RA_ERR_INVALID_ARG, "bad dtype");
  if ((rc = check_scale(scale))) return rc;
  if ((rc = check_ring(s, P, dtype))) return rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(lse, "lse")))
    return rc;
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (dtype == RA_F32) {
    if (s.d != 32 && s.d != 64 && s.d != 128)
      return fail(RA_ERR_UNSUPPORTED, "fp32 path supports d in {32, 64, 128} (got %d)", s.d);
    SimtFwdArgs a{};
    a.q = static_cast<const float*>(q);
    a.k = static_cast<const float*>(k);
    a.v = static_cast<const float*>(v);
    a.B = s.B; a.Nq = s.Nq; a.Nkv = s.Nkv; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d;
    a.ql = s.ql; a.kvl = s.kvl;
    a.scale = scale; a.causal = causal;
    a.P = P; a.S = s.Nq / P; a.striped = striped; a.host_len = host_len;
    a.o_out = o; a.o_dtype = o_dtype; a.lse = lse;
    TimedLaunch tl(RA_KERNEL_FWD_F32, cs);
    cudaError_t e = launch_simt_fwd(a, cs);
    return e == cudaSuccess ? RA_OK : cuda_fail(e, "fp32 ring forward launch");
  }
  if ((rc = check_tc(s, dtype))) return rc;
  const size_t need = ra_ring_fwd_workspace_bytes(dtype, shape, P);
  if (!workspace || ws_bytes < need)
    return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  unsigned int* sched = static_cast<unsigned int*>(workspace);
  cudaError_t me = cudaMemsetAsync(sched, 0, 256, cs);
  if (me != cudaSuccess) return cuda_fail(me, "zero unit counter");
  const void* v16 = v;
  if (dtype == RA_BF16) {
    void* vcopy = static_cast<char*>(workspace) + 256;
    cudaError_t e = launch_to_f16(v, RA_BF16, s.kvl, vcopy, s.B, s.Nkv, s.Hkv, s.d, st, cs);
    if (e != cudaSuccess) return cuda_fail(e, "v -> fp16 launch");
    v16 = vcopy;
  }
  TcFwdArgs a;
  memset(&a, 0, sizeof a);
  const int bf = dtype == RA_BF16;
  if ((rc = make_map(&a.tm_q, q, bf, s.B, s.Nq, s.Hq, s.d, s.ql))) return rc;
  if ((rc = make_map(&a.tm_k, k, bf, s.B, s.Nkv, s.Hkv, s.d, s.kvl))) return rc;
  if ((rc = make_map(&a.tm_v, v16, 0, s.B, s.Nkv, s.Hkv, s.d,
                     dtype == RA_BF16 ? packed_lay(s.Nkv, s.Hkv, s.d) : s.kvl)))
    return rc;
  a.qk_bf16 = bf;
  a.B = s.B; a.Nq = s.Nq; a.Nkv = s.Nkv; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal;
  a.ring_P = P; a.ring_S = s.Nq / P; a.T_m = div_magic((unsigned)(a.ring_S / 128)); a.mode = 0; a.precise = precise; a.striped = striped;
  a.host_len = host_len;
  if (host_len) {  // padded rows: O = 0, LSE = -inf (the kernel skips them)
    cudaError_t fe = launch_fill_padding(o, o_dtype, s.ql, s.B, s.Nq, s.Hq, s.d, P, host_len, lse, cs);
    if (fe != cudaSuccess) return cuda_fail(fe, "padding fill launch");
  }
  a.o_out = o; a.o_dtype = o_dtype; a.ol = s.ql; a.lse = lse;
  a.status = st;
  a.wait_limit_ns = wait_limit_ns();
  a.log = visit_log();
  const int T = a.ring_S / 128;
  a.num_units = s.B * s.Hq * P * ((T + 1) / 2);
  a.sched = sched;
  TimedLaunch tl(RA_KERNEL_FWD_TC, cs);
  cudaError_t e = launch_tc_fwd(a, device_sms(), cs);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "tensor-core ring forward launch");
}

// Backward workspace: D [B,Hq,N] fp32 | LSE*log2e [B,Hq,N] fp32 |
// dq_acc [B,N,Hq,d] fp32 | unit counter (256 bytes, zeroed with dq_acc) |
// fp16 copies of q, k, v, dO (16-bit dtypes that are not already fp16).
struct BwdWs {
  size_t D, lse2, dq, sched, q16, k16, v16, do16, total;
};
static BwdWs bwd_layout(int dtype, const ra_shape& sh) {
  BwdWs w{};
  const size_t qel = (size_t)sh.B * sh.N_q * sh.Hq * sh.d;
  const size_t kvel = (size_t)sh.B * sh.N_kv * sh.Hkv * sh.d;
  size_t off = 0;
  w.D = off; off += align256((size_t)sh.B * sh.Hq * sh.N_q * 4);
  if (dtype != RA_F32) {
    w.lse2 = off; off += align256((size_t)sh.B * sh.Hq * sh.N_q * 4);
    w.dq = off; off += align256(qel * 4);
    w.sched = off; off += 256;
    if (dtype == RA_BF16) {
      w.q16 = off; off += align256(qel * 2);
      w.k16 = off; off += align256(kvel * 2);
      w.v16 = off; off += align256(kvel * 2);
      w.do16 = off; off += align256(qel * 2);
    }
  }
  w.total = off;
  return w;
}

size_t ra_ring_bwd_workspace_bytes(ra_dtype dtype, ra_dtype grad_dtype, ra_shape shape, int P) {
  (void)grad_dtype;
  (void)P;
  if (shape.B < 1 || shape.N_q < 1 || shape.N_kv < 1 || shape.Hq < 1 || shape.Hkv < 1 || shape.d < 1) return 0;
  return bwd_layout(dtype, shape).total;
}

static int ring_bwd_impl(const void* q, const void* k, const void* v, const void* o, ra_dtype o_dtype,
                         const void* dO, const float* lse, ra_dtype dtype, ra_shape shape, int P,
                         int flags, float scale, void* dq, void* dk, void* dv, ra_dtype grad_dtype,
                         void* workspace, size_t ws_bytes, void* stream, const int* host_len) {
  const int causal = (flags & RA_CAUSAL) != 0, precise = (flags & RA_PRECISE) != 0;
  const int striped = causal && (flags & RA_STRIPED) != 0;
  if (flags & ~(RA_CAUSAL | RA_PRECISE | RA_STRIPED))
    return fail(RA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  if (host_len && striped)
    return fail(RA_ERR_INVALID_ARG, "RA_STRIPED does not combine with per-host lengths");
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if (!valid_dtype(dtype) || !valid_dtype(o_dtype) || !valid_dtype(grad_dtype))
    return fail(RA_ERR_INVALID_ARG, "bad dtype");
  if ((rc = check_scale(scale))) return rc;
  if ((rc = check_ring(s, P, dtype))) return rc;
  if ((rc = check_ptr(q, "q")) || (rc = check_ptr(k, "k")) || (rc = check_ptr(v, "v")) ||
      (rc = check_ptr(o, "o")) || (rc = check_ptr(dO, "dO")) || (rc = check_ptr(lse, "lse")) ||
      (rc = check_ptr(dq, "dq")) || (rc = check_ptr(dk, "dk")) || (rc = check_ptr(dv, "dv")))
    return rc;
  const BwdWs w = bwd_layout(dtype, shape);
  if (!workspace || ws_bytes < w.total)
    return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", w.total, ws_bytes);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  float* Dv = reinterpret_cast<float*>(ws + w.D);
  if (dtype == RA_F32) {
    if (s.d != 32 && s.d != 64 && s.d != 128)
      return fail(RA_ERR_UNSUPPORTED, "fp32 path supports d in {32, 64, 128} (got %d)", s.d);
    cudaError_t e = launch_bwd_dot(dO, RA_F32, o, o_dtype, s.ql, Dv, nullptr, nullptr, s.B, s.Nq,
                                   s.Hq, s.d, cs);
    if (e != cudaSuccess) return cuda_fail(e, "bwd D launch");
    SimtBwdArgs a{};
    a.q = static_cast<const float*>(q);
    a.k = static_cast<const float*>(k);
    a.v = static_cast<const float*>(v);
    a.dO = static_cast<const float*>(dO);
    a.lse = lse;
    a.Dvec = Dv;
    a.B = s.B; a.N = s.Nq; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d;
    a.ql = s.ql; a.kvl = s.kvl;
    a.scale = scale; a.causal = causal;
    a.P = P; a.S = s.Nq / P; a.striped = striped; a.host_len = host_len;
    a.dq = dq; a.dk = dk; a.dv = dv; a.grad_dtype = grad_dtype;
    {
      TimedLaunch tl(RA_KERNEL_BWD_F32, cs);
      e = launch_simt_bwd(a, cs);
    }
    return e == cudaSuccess ? RA_OK : cuda_fail(e, "fp32 ring backward launch");
  }
  if ((rc = check_tc(s, dtype))) return rc;
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2);
  cudaError_t e = launch_bwd_dot(dO, dtype, o, o_dtype, s.ql, Dv, lse, lse2, s.B, s.Nq, s.Hq,
                                 s.d, cs);
  if (e != cudaSuccess) return cuda_fail(e, "bwd D launch");
  const void *q16 = q, *k16 = k, *v16 = v, *do16 = dO;
  Lay q16_l = s.ql, kv16_l = s.kvl;
  if (dtype == RA_BF16) {
    q16 = ws + w.q16; k16 = ws + w.k16; v16 = ws + w.v16; do16 = ws + w.do16;
    q16_l = packed_lay(s.Nq, s.Hq, s.d);
    kv16_l = packed_lay(s.Nkv, s.Hkv, s.d);
    if ((e = launch_to_f16(q, RA_BF16, s.ql, ws + w.q16, s.B, s.Nq, s.Hq, s.d, st, cs)) != cudaSuccess ||
        (e = launch_to_f16(k, RA_BF16, s.kvl, ws + w.k16, s.B, s.Nkv, s.Hkv, s.d, st, cs)) != cudaSuccess ||
        (e = launch_to_f16(v, RA_BF16, s.kvl, ws + w.v16, s.B, s.Nkv, s.Hkv, s.d, st, cs)) != cudaSuccess ||
        (e = launch_to_f16(dO, RA_BF16, s.ql, ws + w.do16, s.B, s.Nq, s.Hq, s.d, st, cs)) != cudaSuccess)
      return cuda_fail(e, "fp16 operand copy launch");
  }
  float* dq_acc = reinterpret_cast<float*>(ws + w.dq);
  e = cudaMemsetAsync(dq_acc, 0, w.sched + 256 - w.dq, cs);  // and the unit counter
  if (e != cudaSuccess) return cuda_fail(e, "zero dq accumulator");
  TcBwdArgs a;
  memset(&a, 0, sizeof a);
  if ((rc = make_map(&a.tm_q, q16, 0, s.B, s.Nq, s.Hq, s.d, q16_l)) ||
      (rc = make_map(&a.tm_do, do16, 0, s.B, s.Nq, s.Hq, s.d, q16_l)) ||
      (rc = make_map(&a.tm_k, k16, 0, s.B, s.Nkv, s.Hkv, s.d, kv16_l)) ||
      (rc = make_map(&a.tm_v, v16, 0, s.B, s.Nkv, s.Hkv, s.d, kv16_l)) ||
      (rc = make_map_f32(&a.tm_dq, dq_acc, s.B, s.Nq, s.Hq, s.d)))
    return rc;
  a.B = s.B; a.N = s.Nq; a.Hq = s.Hq; a.Hkv = s.Hkv; a.d = s.d;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal;
  a.ring_P = P; a.ring_S = s.Nq / P; a.T_m = div_magic((unsigned)(a.ring_S / 128)); a.P_m = div_magic((unsigned)P);
  a.precise = precise; a.striped = striped;
  a.host_len = host_len;
  if (host_len) {  // padded key rows: dK = dV = 0 (the kernel skips wholly padded key tiles)
    cudaError_t fe = launch_fill_padding(dk, grad_dtype, s.kvl, s.B, s.Nkv, s.Hkv, s.d, P, host_len, nullptr, cs);
    if (fe == cudaSuccess)
      fe = launch_fill_padding(dv, grad_dtype, s.kvl, s.B, s.Nkv, s.Hkv, s.d, P, host_len, nullptr, cs);
    if (fe != cudaSuccess) return cuda_fail(fe, "padding fill launch");
  }
  a.lse = lse2; a.Dvec = Dv; a.dq_acc = dq_acc;
  a.dk = dk; a.dv = dv; a.grad_dtype = grad_dtype; a.kvl = s.kvl;
  a.status = st;
  a.wait_limit_ns = wait_limit_ns();
  a.log = visit_log();
  a.num_units = s.B * s.Hkv * (s.Nkv / 128);
  a.sched = reinterpret_cast<unsigned int*>(ws + w.sched);
  {
    TimedLaunch tl(RA_KERNEL_BWD_TC, cs);
    e = launch_tc_bwd(a, device_sms(), cs);
  }
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core ring backward launch");
  e = launch_f32_to(dq_acc, dq, grad_dtype, s.ql, s.B, s.Nq, s.Hq, s.d, scale, cs);
  return e == cudaSuccess ? RA_OK : cuda_fail(e, "dq conversion launch");
}

int ra_ring_fwd(const void* q, const void* k, const void* v, ra_dtype dtype, ra_shape shape,
                int P, int flags, float scale, void* o, ra_dtype o_dtype, float* lse,
                void* workspace, size_t ws_bytes, void* stream) {
  return ring_fwd_impl(q, k, v, dtype, shape, P, flags, scale, o, o_dtype, lse, workspace, ws_bytes,
                       stream, nullptr);
}

int ra_ring_bwd(const void* q, const void* k, const void* v, const void* o, ra_dtype o_dtype,
                const void* dO, const float* lse, ra_dtype dtype, ra_shape shape, int P,
                int flags, float scale, void* dq, void* dk, void* dv, ra_dtype grad_dtype,
                void* workspace, size_t ws_bytes, void* stream) {
  return ring_bwd_impl(q, k, v, o, o_dtype, dO, lse, dtype, shape, P, flags, scale, dq, dk, dv,
                       grad_dtype, workspace, ws_bytes, stream, nullptr);
}

int ra_ring_fwd_varlen(const void* q, const void* k, const void* v, ra_dtype dtype, ra_shape shape,
                       int P, const int* host_len, int flags, float scale, void* o, ra_dtype o_dtype,
                       float* lse, void* workspace, size_t ws_bytes, void* stream) {
  if (!host_len || (reinterpret_cast<uintptr_t>(host_len) & 3u))
    return fail(RA_ERR_INVALID_ARG, "host_len must be a non-NULL, 4-byte aligned device array");
  return ring_fwd_impl(q, k, v, dtype, shape, P, flags, scale, o, o_dtype, lse, workspace, ws_bytes,
                       stream, host_len);
}

int ra_ring_bwd_varlen(const void* q, const void* k, const void* v, const void* o, ra_dtype o_dtype,
                       const void* dO, const float* lse, ra_dtype dtype, ra_shape shape, int P,
                       const int* host_len, int flags, float scale, void* dq, void* dk, void* dv,
                       ra_dtype grad_dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (!host_len || (reinterpret_cast<uintptr_t>(host_len) & 3u))
    return fail(RA_ERR_INVALID_ARG, "host_len must be a non-NULL, 4-byte aligned device array");
  return ring_bwd_impl(q, k, v, o, o_dtype, dO, lse, dtype, shape, P, flags, scale, dq, dk, dv,
                       grad_dtype, workspace, ws_bytes, stream, host_len);
}

#pragma GCC visibility pop
}  // extern "C"

// ------------------------------------------------ blockwise feed-forward layer
namespace ra {
namespace {

struct FfnShape {
  long long T;
  int dm, dh, block;
};

int check_ffn(ra_dtype dtype, long long T, int d_model, int d_hidden, int block, FfnShape* out) {
  if (dtype != RA_BF16 && dtype != RA_F16)
    return fail(RA_ERR_UNSUPPORTED, "the feed-forward path takes bf16 or fp16 operands");
  if (T < 1 || d_model < 1 || d_hidden < 1 || block < 1)
    return fail(RA_ERR_INVALID_ARG, "non-positive feed-forward size (T=%lld d_model=%d d_hidden=%d block=%d)", T,
                d_model, d_hidden, block);
  if (d_model % 256 || d_hidden % 256)
    return fail(RA_ERR_UNSUPPORTED, "d_model and d_hidden must be multiples of 256 (got %d, %d)", d_model, d_hidden);
  if (T % 128 || block % 128)
    return fail(RA_ERR_UNSUPPORTED, "T and block must be multiples of 128 (got %lld, %d)", T, block);
  if (T >= (1ll << 31) || d_model > 65536 || d_hidden > 262144)
    return fail(RA_ERR_INVALID_ARG, "feed-forward size too large");
  *out = FfnShape{T, d_model, d_hidden, (int)(block < T ? block : T)};
  return RA_OK;
}

// per-block 16-bit scratch: hidden activations a, GELU'(h), dH
struct FfnWs {
  size_t a, g, dh, total;
};
FfnWs ffn_layout(const FfnShape& s, bool bwd) {
  FfnWs w{};
  const size_t blk = align256((size_t)s.block * s.dh * 2);
  w.a = 0;
  w.g = blk;
  w.dh = 2 * blk;
  w.total = bwd ? 3 * blk : blk;
  return w;
}

struct GemmPlan {
  int rc = RA_OK;
  cudaStream_t st;
  int bf16;
  int* status;
  int sms;
  // a second problem run in the same launch (same K, majorness and epilogue)
  struct Second {
    const void* A;
    long long a_rows, a_cols;
    const void* B;
    long long b_rows, b_cols;
    int M, N;
    void* c;
    long long ldc;
  };
  // C[M, N] = epi(A B^T); a_rows/b_rows are the row counts of the stored matrices
  int run(const void* A, long long a_rows, long long a_cols, int a_mn, const void* B, long long b_rows,
          long long b_cols, int b_mn, int M, int N, int K, int epi, void* c, long long ldc, int c_dtype,
          void* c2 = nullptr, const void* aux = nullptr, const Second* second = nullptr) {
    if (rc) return rc;
    GemmArgs g;
    memset(&g, 0, sizeof g);
    if ((rc = make_map_2d(&g.tm_a, A, bf16, a_rows, a_cols, a_cols, a_mn ? 64 : 128)) ||
        (rc = make_map_2d(&g.tm_b, B, bf16, b_rows, b_cols, b_cols, b_mn ? 64 : 256)))
      return rc;
    g.M = M; g.N = N; g.K = K;
    g.a_mn = a_mn; g.b_mn = b_mn; g.ab_bf16 = bf16;
    g.epi = epi; g.c = c; g.ldc = ldc; g.c_dtype = c_dtype; g.c2 = c2; g.aux = aux;
    g.groups = 1;
    if (second) {
      g.groups = 2;
      if ((rc = make_map_2d(&g.tm_a2, second->A, bf16, second->a_rows, second->a_cols, second->a_cols,
                            a_mn ? 64 : 128)) ||
          (rc = make_map_2d(&g.tm_b2, second->B, bf16, second->b_rows, second->b_cols, second->b_cols,
                            b_mn ? 64 : 256)))
        return rc;
      g.M2 = second->M; g.N2 = second->N; g.c_g2 = second->c; g.ldc_g2 = second->ldc;
    }
    g.status = status;
    g.wait_limit_ns = wait_limit_ns();
    cudaError_t e;
    {
      TimedLaunch tl(RA_KERNEL_GEMM_TC, st);
      e = launch_tc_gemm(g, sms, st);
    }
    if (e != cudaSuccess) rc = cuda_fail(e, "tensor-core GEMM launch");
    return rc;
  }
};

int ffn_common(const void* x, const void* w1, const void* w2, ra_dtype dtype, long long T, int d_model,
               int d_hidden, int block, void* workspace, size_t ws_bytes, bool bwd, FfnShape* s, FfnWs* w,
               int** st) {
  int rc;
  if ((rc = check_ffn(dtype, T, d_model, d_hidden, block, s))) return rc;
  if ((rc = check_ptr(x, "x")) || (rc = check_ptr(w1, "w1")) || (rc = check_ptr(w2, "w2"))) return rc;
  *w = ffn_layout(*s, bwd);
  if (!workspace || ws_bytes < w->total)
    return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", w->total, ws_bytes);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  if ((rc = status_ptr(st))) return rc;
  if (!device_is_sm103()) return fail(RA_ERR_UNSUPPORTED, "tensor-core kernels are built for sm_103a only");
  return RA_OK;
}

}  // namespace
}  // namespace ra

extern "C" {
#pragma GCC visibility push(default)

size_t ra_ffn_workspace_bytes(ra_dtype dtype, long long T, int d_model, int d_hidden, int block, int backward) {
  FfnShape s;
  if (check_ffn(dtype, T, d_model, d_hidden, block, &s)) return 0;
  return ffn_layout(s, backward != 0).total;
}

int ra_ffn_fwd(const void* x, const void* w1, const void* w2, ra_dtype dtype, long long T, int d_model,
               int d_hidden, int block, void* y, ra_dtype y_dtype, void* workspace, size_t ws_bytes, void* stream) {
  FfnShape s;
  FfnWs w;
  int* st;
  int rc = ffn_common(x, w1, w2, dtype, T, d_model, d_hidden, block, workspace, ws_bytes, false, &s, &w, &st);
  if (rc) return rc;
  if (!valid_dtype(y_dtype)) return fail(RA_ERR_INVALID_ARG, "bad y dtype");
  if ((rc = check_ptr(y, "y"))) return rc;
  GemmPlan g;
  g.st = static_cast<cudaStream_t>(stream);
  g.bf16 = dtype == RA_BF16;
  g.status = st;
  g.sms = device_sms();
  char* ws = static_cast<char*>(workspace);
  const size_t es = 2, ys = dtype_size(y_dtype);
  for (long long t0 = 0; t0 < s.T && !g.rc; t0 += s.block) {
    const int Mb = (int)(s.T - t0 < s.block ? s.T - t0 : s.block);
    const char* xb = static_cast<const char*>(x) + (size_t)t0 * s.dm * es;
    // a = GELU(x W1^T) for this block of tokens only
    g.run(xb, Mb, s.dm, 0, w1, s.dh, s.dm, 0, Mb, s.dh, s.dm, GEMM_GELU, ws + w.a, s.dh, dtype);
    // y = a W2^T
    g.run(ws + w.a, Mb, s.dh, 0, w2, s.dm, s.dh, 0, Mb, s.dm, s.dh, GEMM_STORE,
          static_cast<char*>(y) + (size_t)t0 * s.dm * ys, s.dm, y_dtype);
  }
  return g.rc;
}

int ra_ffn_bwd(const void* x, const void* w1, const void* w2, const void* dy, ra_dtype dtype, long long T,
               int d_model, int d_hidden, int block, void* dx, ra_dtype dx_dtype, float* dw1, float* dw2,
               void* workspace, size_t ws_bytes, void* stream) {
  FfnShape s;
  FfnWs w;
  int* st;
  int rc = ffn_common(x, w1, w2, dtype, T, d_model, d_hidden, block, workspace, ws_bytes, true, &s, &w, &st);
  if (rc) return rc;
  if (!valid_dtype(dx_dtype)) return fail(RA_ERR_INVALID_ARG, "bad dx dtype");
  if ((rc = check_ptr(dy, "dy")) || (rc = check_ptr(dx, "dx")) || (rc = check_ptr(dw1, "dw1")) ||
      (rc = check_ptr(dw2, "dw2")))
    return rc;
  GemmPlan g;
  g.st = static_cast<cudaStream_t>(stream);
  g.bf16 = dtype == RA_BF16;
  g.status = st;
  g.sms = device_sms();
  char* ws = static_cast<char*>(workspace);
  const size_t es = 2, xs = dtype_size(dx_dtype);
  cudaError_t e = cudaMemsetAsync(dw1, 0, (size_t)s.dh * s.dm * 4, g.st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, (size_t)s.dm * s.dh * 4, g.st);
  if (e != cudaSuccess) return cuda_fail(e, "zero weight gradients");
  for (long long t0 = 0; t0 < s.T && !g.rc; t0 += s.block) {
    const int Mb = (int)(s.T - t0 < s.block ? s.T - t0 : s.block);
    const char* xb = static_cast<const char*>(x) + (size_t)t0 * s.dm * es;
    const char* dyb = static_cast<const char*>(dy) + (size_t)t0 * s.dm * es;
    // recompute the block's hidden activations: a = GELU(h), g = GELU'(h), h = x W1^T
    g.run(xb, Mb, s.dm, 0, w1, s.dh, s.dm, 0, Mb, s.dh, s.dm, GEMM_GELU2, ws + w.a, s.dh, dtype, ws + w.g);
    // dH = (dy W2) * GELU'(h)   (W2 [dm, dh] read as a [K, N] matrix: MN-major)
    g.run(dyb, Mb, s.dm, 0, w2, s.dm, s.dh, 1, Mb, s.dh, s.dm, GEMM_MUL, ws + w.dh, s.dh, dtype, nullptr,
          ws + w.g);
    // dx = dH W1   (W1 [dh, dm] as [K, N]: MN-major)
    g.run(ws + w.dh, Mb, s.dh, 0, w1, s.dh, s.dm, 1, Mb, s.dm, s.dh, GEMM_STORE,
          static_cast<char*>(dx) + (size_t)t0 * s.dm * xs, s.dm, dx_dtype);
    // dW2 += dy^T a   (M = d_model, N = d_hidden, K = the block's tokens; both operands MN-major)
    // and, in the same launch, dW1 += dH^T x   (M = d_hidden, N = d_model): each alone has
    // too few 128 x 256 tiles to keep the last wave of SMs busy
    const GemmPlan::Second dw1_prob{ws + w.dh, Mb, s.dh, xb, Mb, s.dm, s.dh, s.dm, dw1, s.dm};
    g.run(dyb, Mb, s.dm, 1, ws + w.a, Mb, s.dh, 1, s.dm, s.dh, Mb, GEMM_ACC, dw2, s.dh, RA_F32, nullptr, nullptr,
          &dw1_prob);
  }
  return g.rc;
}

#pragma GCC visibility pop
}  // extern "C"

// ----------------------------------------------------- one step from host memory
namespace ra {
namespace {

// Device workspace of ra_ring_step_host: device copies of the inputs and
// outputs (packed [B, N, H, d]; LSE [B, Hq, N]) and the forward and backward
// workspaces.
struct HostWs {
  size_t q, k, v, dO, o, lse, dq, dk, dv, fwd, bwd, total;
};
HostWs host_layout(int dtype, int o_dtype, int grad_dtype, const ra_shape& sh, int P) {
  HostWs w{};
  const size_t qel = (size_t)sh.B * sh.N_q * sh.Hq * sh.d, kvel = (size_t)sh.B * sh.N_kv * sh.Hkv * sh.d;
  ra_shape packed = sh;
  packed.q_bstride = packed.q_rstride = packed.q_hstride = 0;
  packed.kv_bstride = packed.kv_rstride = packed.kv_hstride = 0;
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  const size_t es = dtype_size(dtype), gs = dtype_size(grad_dtype);
  w.q = take(qel * es);
  w.k = take(kvel * es);
  w.v = take(kvel * es);
  w.dO = take(qel * es);
  w.o = take(qel * dtype_size(o_dtype));
  w.lse = take((size_t)sh.B * sh.Hq * sh.N_q * 4);
  w.dq = take(qel * gs);
  w.dk = take(kvel * gs);
  w.dv = take(kvel * gs);
  w.fwd = take(ra_ring_fwd_workspace_bytes((ra_dtype)dtype, packed, P));
  w.bwd = take(ra_ring_bwd_workspace_bytes((ra_dtype)dtype, (ra_dtype)grad_dtype, packed, P));
  w.total = off;
  return w;
}

// Side streams of ra_ring_step_host, one pair per device, created on first
// use and kept for the life of the process.
struct SideStreams {
  std::mutex mu;
  cudaStream_t in[kMaxDevices] = {}, out[kMaxDevices] = {};
};
SideStreams& side_streams() {
  static SideStreams s;
  return s;
}
int get_side_streams(cudaStream_t* in, cudaStream_t* out) {
  int dev;
  int rc = current_device(&dev);
  if (rc) return rc;
  SideStreams& s = side_streams();
  std::lock_guard<std::mutex> lk(s.mu);
  if (!s.in[dev]) {
    cudaError_t e = cudaStreamCreateWithFlags(&s.in[dev], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.out[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      s.in[dev] = s.out[dev] = nullptr;
      return cuda_fail(e, "create side streams");
    }
  }
  *in = s.in[dev];
  *out = s.out[dev];
  return RA_OK;
}

// Copies B batches of `batch` elements between a buffer with batch stride
// `src_bs` and one with batch stride `dst_bs` (elements of `es` bytes).
cudaError_t copy_batches(void* dst, long long dst_bs, const void* src, long long src_bs, int B,
                         long long batch, size_t es, cudaStream_t st) {
  if (dst_bs == batch && src_bs == batch)
    return cudaMemcpyAsync(dst, src, (size_t)B * batch * es, cudaMemcpyDefault, st);
  for (int b = 0; b < B; ++b) {
    cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dst) + (size_t)b * dst_bs * es,
                                    static_cast<const char*>(src) + (size_t)b * src_bs * es,
                                    (size_t)batch * es, cudaMemcpyDefault, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

struct Events {
  cudaEvent_t e[4] = {};
  ~Events() {
    for (cudaEvent_t x : e)
      if (x) cudaEventDestroy(x);  // released once the recorded work completes
  }
};

}  // namespace
}  // namespace ra

extern "C" {
#pragma GCC visibility push(default)

size_t ra_ring_step_host_workspace_bytes(ra_dtype dtype, ra_dtype o_dtype, ra_dtype grad_dtype,
                                         ra_shape shape, int P) {
  if (shape.B < 1 || shape.N_q < 1 || shape.N_kv < 1 || shape.Hq < 1 || shape.Hkv < 1 || shape.d < 1 ||
      !valid_dtype(dtype) || !valid_dtype(o_dtype) || !valid_dtype(grad_dtype))
    return 0;
  return host_layout(dtype, o_dtype, grad_dtype, shape, P).total;
}

int ra_ring_step_host(const void* q, const void* k, const void* v, const void* dO, ra_dtype dtype,
                      ra_shape shape, int P, int flags, float scale, void* o, ra_dtype o_dtype,
                      float* lse, void* dq, void* dk, void* dv, ra_dtype grad_dtype, void* workspace,
                      size_t ws_bytes, void* stream) {
  // everything the forward and backward would reject is rejected before any
  // copy is enqueued
  if (flags & ~(RA_CAUSAL | RA_PRECISE | RA_STRIPED))
    return fail(RA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  Shape s;
  int rc;
  if ((rc = check_shape(shape, &s))) return rc;
  if (!valid_dtype(dtype) || !valid_dtype(o_dtype) || !valid_dtype(grad_dtype))
    return fail(RA_ERR_INVALID_ARG, "bad dtype");
  if ((rc = check_scale(scale))) return rc;
  if ((rc = check_ring(s, P, dtype))) return rc;
  const void* ins[4] = {q, k, v, dO};
  const char* in_names[4] = {"q", "k", "v", "dO"};
  for (int i = 0; i < 4; ++i)
    if (!ins[i]) return fail(RA_ERR_INVALID_ARG, "%s is NULL", in_names[i]);
  if (!o || !lse || !dq || !dk || !dv) return fail(RA_ERR_INVALID_ARG, "an output pointer is NULL");
  if (!is_packed(s.ql, s.Nq, s.Hq, s.d) || !is_packed(s.kvl, s.Nkv, s.Hkv, s.d))
    return fail(RA_ERR_UNSUPPORTED,
                "ra_ring_step_host takes host tensors with packed rows (row stride H*d, head stride d); "
                "batch strides may be any");
  const HostWs w = host_layout(dtype, o_dtype, grad_dtype, shape, P);
  if (!workspace || ws_bytes < w.total)
    return fail(RA_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", w.total, ws_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(RA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  int* st;
  if ((rc = status_ptr(&st))) return rc;
  if (dtype == RA_F32) {
    if (s.d != 32 && s.d != 64 && s.d != 128)
      return fail(RA_ERR_UNSUPPORTED, "fp32 path supports d in {32, 64, 128} (got %d)", s.d);
  } else {
    Shape packed = s;
    packed.ql = packed_lay(s.Nq, s.Hq, s.d);
    packed.kvl = packed_lay(s.Nkv, s.Hkv, s.d);
    if ((rc = check_tc(packed, dtype))) return rc;
  }
  cudaStream_t main_st = static_cast<cudaStream_t>(stream), in_st, out_st;
  if ((rc = get_side_streams(&in_st, &out_st))) return rc;
  Events ev;
  for (cudaEvent_t& e : ev.e) {
    cudaError_t err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (err != cudaSuccess) return cuda_fail(err, "cudaEventCreateWithFlags");
  }
  char* ws = static_cast<char*>(workspace);
  const long long qel = (long long)s.Nq * s.Hq * s.d, kvel = (long long)s.Nkv * s.Hkv * s.d;
  const size_t es = dtype_size(dtype), gs = dtype_size(grad_dtype);
  ra_shape packed = shape;
  packed.q_bstride = packed.q_rstride = packed.q_hstride = 0;
  packed.kv_bstride = packed.kv_rstride = packed.kv_hstride = 0;
  cudaError_t e;
  // dO travels on the input side stream while q, k, v go up and the forward runs
  if ((e = cudaEventRecord(ev.e[0], main_st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(in_st, ev.e[0], 0)) != cudaSuccess)
    return cuda_fail(e, "dO upload");
  {
    TimedLaunch tl(RA_COPY_H2D, in_st);
    if ((e = copy_batches(ws + w.dO, qel, dO, s.ql.bs, s.B, qel, es, in_st)) != cudaSuccess)
      return cuda_fail(e, "dO upload");
  }
  if ((e = cudaEventRecord(ev.e[1], in_st)) != cudaSuccess) return cuda_fail(e, "dO upload");
  {
    TimedLaunch tl(RA_COPY_H2D, main_st);
    if ((e = copy_batches(ws + w.q, qel, q, s.ql.bs, s.B, qel, es, main_st)) != cudaSuccess ||
        (e = copy_batches(ws + w.k, kvel, k, s.kvl.bs, s.B, kvel, es, main_st)) != cudaSuccess ||
        (e = copy_batches(ws + w.v, kvel, v, s.kvl.bs, s.B, kvel, es, main_st)) != cudaSuccess)
      return cuda_fail(e, "q, k, v upload");
  }
  rc = ring_fwd_impl(ws + w.q, ws + w.k, ws + w.v, dtype, packed, P, flags, scale, ws + w.o, o_dtype,
                     reinterpret_cast<float*>(ws + w.lse), ws + w.fwd, w.bwd - w.fwd, stream, nullptr);
  if (rc) return rc;
  // O and LSE travel down on the output side stream while the backward runs
  if ((e = cudaEventRecord(ev.e[2], main_st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(out_st, ev.e[2], 0)) != cudaSuccess)
    return cuda_fail(e, "O, LSE download");
  {
    TimedLaunch tl(RA_COPY_D2H, out_st);
    if ((e = copy_batches(o, s.ql.bs, ws + w.o, qel, s.B, qel, dtype_size(o_dtype), out_st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(lse, ws + w.lse, (size_t)s.B * s.Hq * s.Nq * 4, cudaMemcpyDefault, out_st)) !=
            cudaSuccess)
      return cuda_fail(e, "O, LSE download");
  }
  if ((e = cudaEventRecord(ev.e[3], out_st)) != cudaSuccess) return cuda_fail(e, "O, LSE download");
  if ((e = cudaStreamWaitEvent(main_st, ev.e[1], 0)) != cudaSuccess) return cuda_fail(e, "join dO upload");
  rc = ring_bwd_impl(ws + w.q, ws + w.k, ws + w.v, ws + w.o, o_dtype, ws + w.dO,
                     reinterpret_cast<const float*>(ws + w.lse), dtype, packed, P, flags, scale, ws + w.dq,
                     ws + w.dk, ws + w.dv, grad_dtype, ws + w.bwd, w.total - w.bwd, stream, nullptr);
  if (rc) return rc;
  {
    TimedLaunch tl(RA_COPY_D2H, main_st);
    if ((e = copy_batches(dq, s.ql.bs, ws + w.dq, qel, s.B, qel, gs, main_st)) != cudaSuccess ||
        (e = copy_batches(dk, s.kvl.bs, ws + w.dk, kvel, s.B, kvel, gs, main_st)) != cudaSuccess ||
        (e = copy_batches(dv, s.kvl.bs, ws + w.dv, kvel, s.B, kvel, gs, main_st)) != cudaSuccess)
      return cuda_fail(e, "gradient download");
  }
  if ((e = cudaStreamWaitEvent(main_st, ev.e[3], 0)) != cudaSuccess) return cuda_fail(e, "join O download");
  return RA_OK;
}

#pragma GCC visibility pop
}  // extern "C"
