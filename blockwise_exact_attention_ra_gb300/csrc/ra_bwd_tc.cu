// Backward blockwise attention on the sm_103a tensor cores (tcgen05 + TMEM +
// TMA).
//
// What it computes: the gradients of L = sum(O * dO) for exact attention,
// with the probabilities recomputed from the saved LSE rather than stored
// (activation recomputation; "Ring Attention: Train 1M Tokens on 8GB GPUs in
// 2026", "Building Ring Attention in PyTorch: The 200-Line Version").  Each
// key/value tile keeps its dK, dV accumulators in TMEM while it travels the
// ring: block j visits hosts (j + s) mod P, s = 0, 1, ... (its gradients
// "flow backwards through the ring", section "Gotchas and Failure Modes"),
// skipping hosts wholly before it under a causal mask.  Per visited query
// tile i:
//   S^T  = K Q_i^T                    (recompute)
//   P^T  = exp(scale S^T - LSE_i)     (masked on the diagonal tile)
//   dP^T = V dO_i^T
//   dS^T = P^T * (dP^T - D_i),        D_i = rowsum(dO_i * O_i)
//   dV  += P^T dO_i ;  dK += dS^T Q_i ;  dQ_i += dS K   (dQ reduce-added)
// dK is scaled by `scale` at the end, dQ when it is converted.
//
// CTA organisation (one persistent CTA per SM, 14 warps):
//   warp 0       TMA producer: K, V of the unit; Q_i, dO_i (+ LSE, D slices)
//                through two shared-memory stages
//   warp 1       TMEM allocation; one lane issues every tcgen05.mma
//   warps 2-9    compute: thread = key row; warps 2-5 take query columns
//                0-63, warps 6-9 columns 64-127
//   warps 10-13  dQ: read dQ_i from TMEM (thread = query row), stage it in
//                shared memory and reduce-add it into the fp32 accumulator
//                with TMA (whole 128-byte lines); at the end of a unit write
//                dK, dV
// Shared memory has no room for a dQ buffer, but once dQ_i is complete the
// last MMA that reads dO_i (dV) has completed too, so the dQ warps stage dQ_i
// in that stage's dO buffer, in two rounds of D/2 columns, and hand the dO
// buffer back to the producer once the TMA engine has read the second round.
// Q and dO have separate stage barriers: the Q buffer returns to the producer
// as soon as dK has consumed it, so the next query tile's S MMA never waits
// for a reduction (dO_{i+2} is needed latest in an iteration).  (Per-thread
// red.global of whole rows cost ~6000 cycles per tile in the load/store unit
// and starved the compute warps' shared-memory traffic.)
// TMEM (512 columns): S^T [0,128) (P^T as fp16 written back into columns
// [0,32) and [64,96); dS^T as fp16 into [32,64) and [96,128)), dP^T [128,256)
// (dQ_i reuses [128,128+D)), dK [256,256+D), dV [256+D,256+2D).
// MMA order per iteration: dV(i) dQ(i) dK(i) S(i+1) dP(i+1).  dK takes dS^T
// from TMEM (the S^T columns that P^T leaves free), so of the five products
// only S, dP and dQ read both operands from shared memory; S(i+1) overwrites
// those columns after dK(i), which also leaves the next Q tile's load more
// time; dQ(i) leaves TMEM while dK(i) and S(i+1) run, before dP(i+1) needs
// its columns.
// With PRECISE, dS enters the dK product as two fp16 terms (hi from shared
// memory, lo = fp16(dS - hi) from TMEM columns of dP^T that have already been
// read: [128+64h, 128+64h+32) for query half h), so its rounding drops from
// 2^-12 relative to about 2^-24; dQ keeps the single fp16 term.  That mode
// keeps the order dV(i) S(i+1) dK(i) dQ(i) dP(i+1).
#include <math.h>

#include "ra_device.cuh"

namespace ra {
namespace {

constexpr int kThreads = 448;

template <int D>
struct BwdSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ0 = 2 * kTile;      // Q stage s at kQ0 + s * kTile
  static constexpr int kDO0 = 4 * kTile;     // dO stage s
  static constexpr int kDS = 6 * kTile;      // dS^T, 128 key rows x 128 query columns fp16
  static constexpr int kDSBytes = 128 * 128 * 2;
  static constexpr int kVec0 = kDS + kDSBytes;  // per stage: LSE*log2e [128], D [128]
  static constexpr int kBars = kVec0 + 2 * 1024;
  // kv_full, kv_empty, q_full[2], q_empty[2], s_full, dp_full, ds_full,
  // ds_free, dq_full, dq_free, dkv_full, dkv_free, drain, (unused),
  // do_full[2], do_empty[2], (unused), p_full, unit_full[4], unit_empty[4]
  static constexpr int kNumBars = 30;
  static constexpr int kMisc = kBars + kNumBars * 8;  // TMEM address, abort flag
  static constexpr int kUnits = kMisc + 16;           // unit ring: 4 unit indices
  static constexpr int kUsed = kUnits + 16;
  // at least 120 KB so that one CTA (holding all 512 TMEM columns) occupies an SM
  static constexpr int kBytes = kUsed > 122880 ? kUsed : 122880;
};

struct BwdUnit {
  int b, g, jt;
  int count;  // query tiles per head
  int n_iter; // count * group
  int host, tk, per_block;  // striped layouts: key host, local key tile, query tiles per block
  unsigned long long count_m;  // div_magic(count)
};

// Units are ordered head-major: every resident CTA works on the same
// (batch, key/value head) at a time, so the query tiles, dO tiles and dQ
// accumulator rows they sweep stay in L2 (one head of them is ~128 MB at
// N = 131072).  Within a head the earliest key tiles come first: under a
// causal mask they have the most work.  The CTAs draw units in this order
// from a counter in global memory, so a CTA that finishes early takes the
// next unit instead of running ahead into another head, and the lightest
// units end the launch.
__device__ __forceinline__ int host_len_at(const int* hl, int j, int S);

template <bool STRIPED, bool VARLEN>
__device__ __forceinline__ BwdUnit bwd_unit(const TcBwdArgs& a, int u) {
  BwdUnit r;
  const int nT = a.N / 128;
  const int bg = u / nT;
  r.jt = u % nT;
  r.b = bg / a.Hkv;
  r.g = bg % a.Hkv;
  if (STRIPED) {
    // striped: local key tile tk meets local query tiles tk..T-1 of every host;
    // smallest local tiles (most work) first, across hosts
    const int T = a.ring_S / 128;
    const int idx = u % nT;
    r.tk = idx / a.ring_P;
    r.host = idx % a.ring_P;
    r.jt = r.host * T + r.tk;
    r.per_block = T - r.tk;
    r.count = a.ring_P * r.per_block;
    r.n_iter = r.count * (a.Hq / a.Hkv);
    r.count_m = div_magic((unsigned)r.count);
    return r;
  }
  r.count = a.causal ? nT - r.jt : nT;
  r.n_iter = r.count * (a.Hq / a.Hkv);
  r.count_m = div_magic((unsigned)r.count);
  if (VARLEN) {
    // key tiles wholly in their host's padding do no work (their dK, dV rows
    // were zero-filled beforehand)
    const int T = a.ring_S / 128;
    const int j = div_by(r.jt, a.T_m);
    if ((r.jt - j * T) * 128 >= host_len_at(a.host_len, j, a.ring_S)) r.n_iter = 0;
  }
  return r;
}

// Query head and query tile of iteration it, in ring order.
template <bool STRIPED>
__device__ __forceinline__ void bwd_iter(const TcBwdArgs& a, const BwdUnit& u, int it, int* h,
                                         int* qt) {
  const int group = a.Hq / a.Hkv;
  const int hh = div_by(it, u.count_m), k = it - hh * u.count;
  *h = u.g * group + hh;
  if (STRIPED) {
    // The key tile goes round the ring once per local query tile it meets:
    // lap t takes local query tile tk + t of hosts (j + s) mod P, s = 0..P-1.
    // The CTAs holding the same local key tile of different hosts then read
    // the same P query tiles within P iterations of each other, which keeps
    // those tiles (and their dQ lines) in L2; a host-by-host sweep spreads a
    // tile's readers over the whole unit.  Only rounding depends on the order.
    const int lap = div_by(k, a.P_m);
    int qh = u.host + (k - lap * a.ring_P);  // both < P
    if (qh >= a.ring_P) qh -= a.ring_P;
    *qt = qh * (a.ring_S / 128) + u.tk + lap;
    return;
  }
  if (a.causal) {
    *qt = u.jt + k;
  } else {
    const int nT = a.N / 128;
    const int T = a.ring_S / 128;
    int q = div_by(u.jt, a.T_m) * T + k;  // < 2 nT
    if (q >= nT) q -= nT;
    *qt = q;
  }
}

// Variable host lengths: valid rows of host j (clamped to [0, S]); a query
// tile wholly in its host's padding is skipped by every role.
__device__ __forceinline__ int host_len_at(const int* hl, int j, int S) {
  const int v = __ldg(hl + j);
  return v < 0 ? 0 : (v > S ? S : v);
}
template <bool VARLEN>
__device__ __forceinline__ bool q_tile_valid(const TcBwdArgs& a, int qt) {
  if (!VARLEN) return true;
  const int T = a.ring_S / 128;
  const int i = div_by(qt, a.T_m);
  return (qt - i * T) * 128 < host_len_at(a.host_len, i, a.ring_S);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// TMA reduce-add of one 128-row x 32-column fp32 box from shared memory.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                  int c2, int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          map),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// dQ staging: round r (columns [r*D/2, (r+1)*D/2)) of stage s goes to the
// dO buffer of that stage as D/64 boxes of 32 fp32 columns x 128 rows (16 KB).
template <int D>
__device__ __forceinline__ uint32_t dq_box(int s, int cc) {
  using L = BwdSmem<D>;
  return L::kDO0 + s * L::kTile + cc * 16384;
}

// Ring layouts, one kernel build each: contiguous hosts, striped rows, and
// contiguous hosts with variable valid lengths.
enum { kLayoutContiguous = 0, kLayoutStriped = 1, kLayoutVarlen = 2 };

template <int D, bool PRECISE, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) tc_bwd_kernel(const __grid_constant__ TcBwdArgs a) {
  using L = BwdSmem<D>;
  constexpr bool STRIPED = LAYOUT == kLayoutStriped, VARLEN = LAYOUT == kLayoutVarlen;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) report(a.status, RA_ERR_UNSUPPORTED);
    return;
  }
  const uint32_t bar0 = sbase + L::kBars;
  const uint32_t BAR_KV_FULL = bar0, BAR_KV_EMPTY = bar0 + 8;
  auto bar_q_full = [&](int s) { return bar0 + 16 + 8 * s; };
  auto bar_q_empty = [&](int s) { return bar0 + 32 + 8 * s; };
  auto bar_do_full = [&](int s) { return bar0 + 128 + 8 * s; };
  auto bar_do_empty = [&](int s) { return bar0 + 144 + 8 * s; };
  const uint32_t BAR_P_FULL = bar0 + 168;
  auto bar_unit_full = [&](int s) { return bar0 + 176 + 8 * s; };
  auto bar_unit_empty = [&](int s) { return bar0 + 208 + 8 * s; };
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + L::kUnits);
  const uint32_t BAR_S_FULL = bar0 + 48, BAR_DP_FULL = bar0 + 56, BAR_DS_FULL = bar0 + 64,
                 BAR_DS_FREE = bar0 + 72, BAR_DQ_FULL = bar0 + 80, BAR_DQ_FREE = bar0 + 88,
                 BAR_DKV_FULL = bar0 + 96, BAR_DKV_FREE = bar0 + 104, BAR_DRAIN = bar0 + 112;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(BAR_KV_FULL, 1);
    mbar_init(BAR_KV_EMPTY, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_q_full(s), 1);
      mbar_init(bar_q_empty(s), 1);
      mbar_init(bar_do_full(s), 1);
      mbar_init(bar_do_empty(s), 4);  // one arrival per dQ warp
    }
    mbar_init(BAR_S_FULL, 1);
    mbar_init(BAR_DP_FULL, 1);
    mbar_init(BAR_DS_FULL, 256);
    mbar_init(BAR_DS_FREE, 1);
    mbar_init(BAR_DQ_FULL, 1);
    mbar_init(BAR_DQ_FREE, 128);
    mbar_init(BAR_DKV_FULL, 1);
    mbar_init(BAR_DKV_FREE, 128);
    mbar_init(BAR_DRAIN, 1);
    mbar_init(BAR_P_FULL, 256);
    // the producer draws the CTA's units and passes them on through a ring of
    // four slots; every consumer thread (MMA lane, 256 compute and 128 dQ
    // threads) hands a slot back once it has read it
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar_unit_full(s), 1);
      mbar_init(bar_unit_empty(s), 1 + 256 + 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
    tma_prefetch_desc(&a.tm_do);
    tma_prefetch_desc(&a.tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t lim = a.wait_limit_ns;
  const uint32_t T_S = tmem, T_DP = tmem + 128, T_DK = tmem + 256, T_DV = tmem + 256 + D;
  // The n-th unit of this CTA, as the producer drew it (every role but the
  // producer); false if the wait gave up.
  auto take_unit = [&](int n, int* u) {
    const int slot = n & 3;
    if (!mbar_wait(bar_unit_full(slot), (n >> 2) & 1, abort_flag, a.status, lim)) return false;
    *u = unit_ring[slot];
    mbar_arrive(bar_unit_empty(slot));
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_first();  // one unit reads its K, V tile once
      const uint64_t pol_q = policy_evict_normal();  // shared with the CTAs on nearby key tiles
      uint32_t qd_cnt = 0;
      int q_issued[2] = {0, 0}, do_issued[2] = {0, 0};
      int k = 0;
      bool ok = true;
      // n counts the units this CTA has drawn, k those it has worked on (a
      // key tile wholly in padding is no unit); a draw at or past the last
      // unit ends every role
      for (int n = 0; ok; ++n) {
        const int slot = n & 3;
        if (!mbar_wait(bar_unit_empty(slot), ((n >> 2) & 1) ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
        const int u = (int)atomicAdd(a.sched, 1u);
        unit_ring[slot] = u;
        mbar_arrive(bar_unit_full(slot));
        if (u >= a.num_units) break;
        const BwdUnit bu = bwd_unit<STRIPED, VARLEN>(a, u);
        if (VARLEN && bu.n_iter == 0) continue;
        if (!mbar_wait(BAR_KV_EMPTY, (k & 1) ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR_KV_FULL, 2 * L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sbase + L::kK + c * 16384, &a.tm_k, BAR_KV_FULL, c * 64, bu.g, bu.jt * 128, bu.b, pol_kv);
          tma_load_4d(sbase + L::kV + c * 16384, &a.tm_v, BAR_KV_FULL, c * 64, bu.g, bu.jt * 128, bu.b, pol_kv);
        }
        ++k;
        for (int it = 0; it < bu.n_iter; ++it) {
          int h, qt;
          bwd_iter<STRIPED>(a, bu, it, &h, &qt);
          if (VARLEN && !q_tile_valid<VARLEN>(a, qt)) continue;
          if (a.log.entries) log_visit(a.log, 1u, bu.b * a.Hq + h, qt, bu.jt);
          const int s = qd_cnt & 1;
          const uint32_t par = ((qd_cnt >> 1) & 1) ^ 1;
          if (!mbar_wait(bar_q_empty(s), par, abort_flag, a.status, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_q_full(s), L::kTile + 1024);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sbase + L::kQ0 + s * L::kTile + c * 16384, &a.tm_q, bar_q_full(s), c * 64, h, qt * 128, bu.b, pol_q);
          const long long vrow = ((long long)bu.b * a.Hq + h) * a.N + (long long)qt * 128;
          bulk_load(sbase + L::kVec0 + s * 1024, a.lse + vrow, 512, bar_q_full(s));
          bulk_load(sbase + L::kVec0 + s * 1024 + 512, a.Dvec + vrow, 512, bar_q_full(s));
          q_issued[s] = 1;
          if (!mbar_wait(bar_do_empty(s), par, abort_flag, a.status, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_do_full(s), L::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sbase + L::kDO0 + s * L::kTile + c * 16384, &a.tm_do, bar_do_full(s), c * 64, h, qt * 128, bu.b, pol_q);
          do_issued[s] = 1;
          ++qd_cnt;
        }
      }
      if (*abort_flag) {
        const uint64_t drain = 100000000ull;
        (void)mbar_wait(BAR_KV_FULL, (k - 1) & 1, abort_flag, nullptr, drain);
        for (int s = 0; s < 2; ++s) {
          // phase of the last load issued on stage s (loads alternate stages)
          const uint32_t last = qd_cnt > (uint32_t)s ? ((qd_cnt - 1 - s) & ~1u) + s : 0;
          if (q_issued[s]) (void)mbar_wait(bar_q_full(s), (last >> 1) & 1, abort_flag, nullptr, drain);
          if (do_issued[s]) (void)mbar_wait(bar_do_full(s), (last >> 1) & 1, abort_flag, nullptr, drain);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // S^T = K Q^T, dP^T = V dO^T: A, B K-major (M = keys, N = queries)
      const uint32_t id_kq = idesc_f16(0, 0, 0, 128, 128);
      // dV += P^T dO (A from TMEM), dK += dS^T Q: B MN-major (N = head dim)
      const uint32_t id_acc = idesc_f16(0, 0, 1, 128, D);
      // dQ = dS K: A = dS^T viewed MN-major (M = queries), B = K MN-major
      const uint32_t id_dq = idesc_f16(0, 1, 1, 128, D);
      const uint32_t sK = sbase + L::kK, sV = sbase + L::kV, sDS = sbase + L::kDS;
      uint32_t qd_cnt = 0, ds_cnt = 0, dq_cnt = 0, p_cnt = 0;
      int k = 0;
      bool ok = true;
      // descriptors built once: K-major (LBO unused) and MN-major (LBO = the
      // 16 KB step between 64-column halves) views of each tile
      const uint64_t dK_k = smem_desc_sw128(sK, 16, 1024), dK_mn = smem_desc_sw128(sK, 16384, 1024);
      const uint64_t dV_k = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dS_k = smem_desc_sw128(sDS, 16, 1024), dS_mn = smem_desc_sw128(sDS, 16384, 1024);
      const uint64_t dQ_k0 = smem_desc_sw128(sbase + L::kQ0, 16, 1024), dQ_mn0 = smem_desc_sw128(sbase + L::kQ0, 16384, 1024);
      const uint64_t dO_k0 = smem_desc_sw128(sbase + L::kDO0, 16, 1024), dO_mn0 = smem_desc_sw128(sbase + L::kDO0, 16384, 1024);
      constexpr uint32_t kStageStep = L::kTile >> 4;  // descriptor step between the two stages
      auto mma_nt = [&](uint32_t dt, uint64_t da, uint64_t db) {  // K-major A and B, K = D
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(dt, desc_off(da, off), desc_off(db, off), id_kq, kk > 0);
        }
      };
      auto wait = [&](uint32_t bar, uint32_t par) {
        if (!mbar_wait(bar, par, abort_flag, a.status, lim)) ok = false;
        tc_fence_after();
        return ok;
      };
      // next query tile at or after iteration it that is not wholly padding
      auto next_valid = [&](const BwdUnit& bu, int it) {
        for (; it < bu.n_iter; ++it) {
          int h, qt;
          bwd_iter<STRIPED>(a, bu, it, &h, &qt);
          if (q_tile_valid<VARLEN>(a, qt)) break;
        }
        return it;
      };
      for (int n = 0; ok; ++n) {
        int u;
        if (!take_unit(n, &u) || u >= a.num_units) break;
        const BwdUnit bu = bwd_unit<STRIPED, VARLEN>(a, u);
        if (VARLEN && bu.n_iter == 0) continue;
        if (!wait(BAR_KV_FULL, k & 1)) break;
        // prologue: S(0), dP(0)
        uint32_t s = qd_cnt & 1;
        if (!wait(bar_q_full(s), (qd_cnt >> 1) & 1)) break;
        mma_nt(T_S, dK_k, dQ_k0 + s * kStageStep);
        mma_commit(BAR_S_FULL);
        if (dq_cnt > 0 && !wait(BAR_DQ_FREE, (dq_cnt - 1) & 1)) break;
        if (!wait(bar_do_full(s), (qd_cnt >> 1) & 1)) break;
        mma_nt(T_DP, dV_k, dO_k0 + s * kStageStep);
        mma_commit(BAR_DP_FULL);
        const int it0 = VARLEN ? next_valid(bu, 0) : 0;
        // Per iteration i, in this order:
        //   P(i) stored     -> dV(i) += P^T dO_i
        //   dS(i) stored    -> dQ(i) = dS K, dK(i) += dS^T Q_i (dS^T from TMEM),
        //                      then S(i+1) over the S^T columns
        //   dQ(i) read out  -> dP(i+1) into the dP/dQ columns
        // With RA_PRECISE: P(i) -> dV(i), S(i+1); dS(i) -> dK(i) (its low terms sit
        // in the dP columns), dQ(i); dQ(i) read out -> dP(i+1).
        for (int it = it0, nx; it < bu.n_iter; it = nx) {
          nx = VARLEN ? next_valid(bu, it + 1) : it + 1;
          const uint64_t dQ_mn = dQ_mn0 + s * kStageStep, dO_mn = dO_mn0 + s * kStageStep;
          const bool has_next = nx < bu.n_iter;
          const uint32_t s2 = (qd_cnt + 1) & 1, par2 = ((qd_cnt + 1) >> 1) & 1;
          if (!wait(BAR_P_FULL, p_cnt & 1)) break;
          ++p_cnt;
          if (it == it0 && k > 0 && !wait(BAR_DKV_FREE, (k - 1) & 1)) break;
          // dV += P^T dO_i   (P^T in TMEM: queries 0-63 at columns 0-31, 64-127 at 64-95)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t pa = T_S + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
            mma_ts(T_DV, pa, desc_off(dO_mn, kk * 2048), id_acc, (it > it0 || kk > 0) ? 1u : 0u);
          }
          if (!PRECISE) {
            // dQ(i), then dK(i) with dS^T from TMEM (the S columns P^T leaves
            // free: queries 0-63 at 32-63, 64-127 at 96-127), then S(i+1) over them
            if (!wait(BAR_DS_FULL, ds_cnt & 1)) break;
            ++ds_cnt;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(T_DP, desc_off(dS_mn, kk * 2048), desc_off(dK_mn, kk * 2048), id_dq, kk > 0 ? 1u : 0u);
            mma_commit(BAR_DQ_FULL);
            ++dq_cnt;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t la = T_S + (kk < 4 ? 32 + kk * 8 : 96 + (kk - 4) * 8);
              mma_ts(T_DK, la, desc_off(dQ_mn, kk * 2048), id_acc, (it > it0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar_q_empty(s));  // dK was the last reader of Q_i
            mma_commit(BAR_DS_FREE);
            ++qd_cnt;
            if (has_next) {
              if (!wait(bar_q_full(s2), par2)) break;
              mma_nt(T_S, dK_k, dQ_k0 + s2 * kStageStep);
              mma_commit(BAR_S_FULL);
              if (!wait(BAR_DQ_FREE, (dq_cnt - 1) & 1)) break;
              if (!wait(bar_do_full(s2), par2)) break;
              mma_nt(T_DP, dV_k, dO_k0 + s2 * kStageStep);
              mma_commit(BAR_DP_FULL);
              s = s2;
            } else {
              mma_commit(BAR_DKV_FULL);
              mma_commit(BAR_KV_EMPTY);
            }
            continue;
          }
          if (has_next) {
            if (!wait(bar_q_full(s2), par2)) break;
            mma_nt(T_S, dK_k, dQ_k0 + s2 * kStageStep);
            mma_commit(BAR_S_FULL);
          }
          if (!wait(BAR_DS_FULL, ds_cnt & 1)) break;
          ++ds_cnt;
          // dQ_i = dS K   (the dS^T tile read MN-major: M = queries)
          auto issue_dq = [&]() {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(T_DP, desc_off(dS_mn, kk * 2048), desc_off(dK_mn, kk * 2048), id_dq, kk > 0 ? 1u : 0u);
            mma_commit(BAR_DQ_FULL);  // dO_i (read by dP_i, dV_i) is consumed too: the dQ warps stage dQ_i in its buffer
            ++dq_cnt;
          };
          if (!PRECISE) issue_dq();
          // dK += dS^T Q_i   (dS^T K-major: key rows of 64-query swizzled halves)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(T_DK, desc_off(dS_k, off), desc_off(dQ_mn, kk * 2048), id_acc, (it > it0 || kk > 0) ? 1u : 0u);
          }
          if (PRECISE) {  // + dS_lo^T Q_i, dS_lo^T in TMEM (queries 0-63 at dP columns 0-31, 64-127 at 64-95)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t la = T_DP + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
              mma_ts(T_DK, la, desc_off(dQ_mn, kk * 2048), id_acc, 1u);
            }
          }
          mma_commit(bar_q_empty(s));  // dK was the last reader of Q_i
          if (PRECISE) issue_dq();
          mma_commit(BAR_DS_FREE);
          ++qd_cnt;
          if (has_next) {
            if (!wait(BAR_DQ_FREE, (dq_cnt - 1) & 1)) break;
            if (!wait(bar_do_full(s2), par2)) break;
            mma_nt(T_DP, dV_k, dO_k0 + s2 * kStageStep);
            mma_commit(BAR_DP_FULL);
            s = s2;
          } else {
            mma_commit(BAR_DKV_FULL);
            mma_commit(BAR_KV_EMPTY);
          }
        }
        ++k;
      }
      mma_commit(BAR_DRAIN);
      (void)mbar_wait(BAR_DRAIN, 0, abort_flag, nullptr, 100000000ull);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ compute
    const int half = (warp - 2) / 4;           // query columns [64*half, 64*half + 64)
    const uint32_t quarter = warp & 3;
    const int r = quarter * 32 + lane;         // key row in the tile
    const uint32_t lane_off = (quarter * 32) << 16;
    const uint32_t tS = T_S + lane_off + half * 64;
    const uint32_t tDP = T_DP + lane_off + half * 64;
    const float sl2 = a.scale_log2;
    uint8_t* ds_row = smem + L::kDS + half * 16384 + r * 128;
    uint32_t gi = 0;  // iterations done by this CTA (all units)
    bool ok = true;
    for (int n = 0; ok; ++n) {
      int u;
      if (!take_unit(n, &u) || u >= a.num_units) break;
      const BwdUnit bu = bwd_unit<STRIPED, VARLEN>(a, u);
      // padding: key rows of this tile from kvalid on (variable host lengths)
      int kvalid = 128;
      if (VARLEN) {
        const int T = a.ring_S / 128;
        const int j = div_by(bu.jt, a.T_m);
        kvalid = host_len_at(a.host_len, j, a.ring_S) - (bu.jt - j * T) * 128;
      }
      // kq: position in the current query head's sweep, enough to place the
      // diagonal tiles without the query tile index
      int kq = 0;
      for (int it = 0; it < bu.n_iter; ++it, ++gi) {
        const int kpos = kq;
        if (++kq == bu.count) kq = 0;
        int h = 0, qt = 0;
        if (VARLEN) bwd_iter<STRIPED>(a, bu, it, &h, &qt);
        // padding: query columns of this tile from qvalid on; a tile wholly in
        // padding is skipped by every role
        int qvalid = 128;
        if (VARLEN) {
          const int T = a.ring_S / 128;
          const int i = div_by(qt, a.T_m);
          qvalid = host_len_at(a.host_len, i, a.ring_S) - (qt - i * T) * 128;
          if (qvalid <= 0) { --gi; continue; }
        }
        const int s = gi & 1;
        // -LSE*log2(e) and -D of this stage's query tile, this half's columns
        const float* nlse2 = reinterpret_cast<const float*>(smem + L::kVec0 + s * 1024) + half * 64;
        const float* ndvec = nlse2 + 128;
        if (!mbar_wait(BAR_S_FULL, gi & 1, abort_flag, a.status, lim)) { ok = false; break; }
        // the LSE / D slices of this stage arrived with the Q tile
        if (!mbar_wait(bar_q_full(s), (gi >> 1) & 1, abort_flag, a.status, lim)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[64];
        RA_TMEM_LD32(tS, pr);
        RA_TMEM_LD32(tS + 32, (pr + 32));
        tmem_ld_wait();
        // causal masks: the diagonal tile of a contiguous layout (query column
        // c visible to key row r iff c >= r), the first of the sweep; for a
        // striped layout the same local tile of any host pair, the sweep's
        // first lap (query hosts j, j+1, ... in ring order), strict (c > r)
        // where the query's host index has wrapped below the key's
        const bool pad = VARLEN && (qvalid < 128 || kvalid < 128);
        bool diag;
        int strict = 0;
        if (STRIPED) {
          diag = kpos < a.ring_P;
          strict = bu.host + kpos >= a.ring_P ? 1 : 0;
        } else {
          diag = a.causal && kpos == 0;
        }
        // P^T = exp2(S^T * scale*log2e - LSE*log2e), two columns per fp32x2 FMA
        const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c);
          const float2 a01 = __ffma2_rn(make_float2(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1])), sl2x2,
                                        make_float2(l4.x, l4.y));
          const float2 a23 = __ffma2_rn(make_float2(__uint_as_float(pr[c + 2]), __uint_as_float(pr[c + 3])), sl2x2,
                                        make_float2(l4.z, l4.w));
          pr[c] = __float_as_uint(ex2_approx(a01.x));
          pr[c + 1] = __float_as_uint(ex2_approx(a01.y));
          pr[c + 2] = __float_as_uint(ex2_approx(a23.x));
          pr[c + 3] = __float_as_uint(ex2_approx(a23.y));
        }
        // the masks, only on the tiles that have any: this half's columns below
        // c_lo (causal) or from c_hi on (padded queries), and every column of
        // a padded key row, are zero
        if (diag || pad) {
          const int c_lo = diag ? r + strict - half * 64 : 0;
          const int c_hi = VARLEN ? (r < kvalid ? qvalid - half * 64 : 0) : 64;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < c_lo || c >= c_hi) pr[c] = 0u;
        }
        // P^T (fp16) back into TMEM for the dV MMA
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) pk[j / 2] = pack_half2(__uint_as_float(pr[c + j]), __uint_as_float(pr[c + j + 1]));
          RA_TMEM_ST16(tS + c / 2, pk);
        }
        // P^T is in TMEM (and S^T has been read): the MMA warp may start dV
        // and then overwrite these columns with the next S^T
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR_P_FULL);
        if (!mbar_wait(BAR_DP_FULL, gi & 1, abort_flag, a.status, lim)) { ok = false; break; }
        tc_fence_after();
        // dS^T of the previous iteration must have been consumed by its MMAs
        if (gi > 0 && !mbar_wait(BAR_DS_FREE, (gi - 1) & 1, abort_flag, a.status, lim)) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t dp[32];
          RA_TMEM_LD32(tDP + c, dp);
          tmem_ld_wait();
          uint32_t pk[16];
          uint32_t pl[PRECISE ? 16 : 1];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            // dS = P * (dP - D), two columns per fp32x2 add and multiply
            const float2 ndd = *reinterpret_cast<const float2*>(ndvec + c + j);
            const float2 diff = __fadd2_rn(make_float2(__uint_as_float(dp[j]), __uint_as_float(dp[j + 1])), ndd);
            const float2 ds = __fmul2_rn(make_float2(__uint_as_float(pr[c + j]), __uint_as_float(pr[c + j + 1])), diff);
            const float d0 = ds.x, d1 = ds.y;
            pk[j / 2] = pack_half2(d0, d1);
            if (PRECISE) {
              const float2 hi = unpack_half2(pk[j / 2]);
              pl[j / 2] = pack_half2(d0 - hi.x, d1 - hi.y);
            }
          }
          // dP^T columns [c, c+32) of this half have been read: the lo terms go
          // to its columns [c/2, c/2+16)
          if (PRECISE) RA_TMEM_ST16(tDP + c / 2, pl);
          else RA_TMEM_ST16(tS + 32 + c / 2, pk);  // dS^T for dK, in the S columns P^T leaves free
          // 16-byte chunks (c/8 .. c/8+3) of this row, 128-byte swizzle
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = (c >> 3) + q4;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          }
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR_DS_FULL);
      }
    }
  } else {
    // ------------------------------------------------------------ dQ / epilogue
    const uint32_t quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (quarter * 32) << 16;
    uint32_t dq_cnt = 0;
    int k = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      int u;
      if (!take_unit(n, &u) || u >= a.num_units) break;
      const BwdUnit bu = bwd_unit<STRIPED, VARLEN>(a, u);
      if (VARLEN && bu.n_iter == 0) continue;
      for (int it = 0; it < bu.n_iter; ++it) {
        int h, qt;
        bwd_iter<STRIPED>(a, bu, it, &h, &qt);
        if (VARLEN && !q_tile_valid<VARLEN>(a, qt)) continue;
        if (!mbar_wait(BAR_DQ_FULL, dq_cnt & 1, abort_flag, a.status, lim)) { ok = false; break; }
        ++dq_cnt;
        tc_fence_after();
        const int s = (dq_cnt - 1) & 1;  // the stage that held Q_i, dO_i
        constexpr int HALF = D / 2;           // columns per staging round
        constexpr int BPR = HALF / 32;        // 32-column slabs per round
        // Each warp stages and reduce-adds its own 32 rows (no cross-warp
        // hand-off): slab cc of round rd, row r, 16-byte chunk j at
        // dq_box(s, cc) + r * 128 + ((j ^ (r & 7)) << 4) (128-byte swizzle,
        // the tensor map's layout; a 32-row box starts at row 32 * quarter).
        auto stage = [&](const uint32_t* v) {
#pragma unroll
          for (int cc = 0; cc < BPR; ++cc) {
            uint8_t* box = smem + dq_box<D>(s, cc) + r * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(box + ((j ^ (r & 7)) << 4)) =
                  make_uint4(v[32 * cc + 4 * j], v[32 * cc + 4 * j + 1], v[32 * cc + 4 * j + 2], v[32 * cc + 4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
        };
        auto reduce = [&](int rd) {  // lane 0: this warp's rows of round rd
#pragma unroll
          for (int cc = 0; cc < BPR; ++cc)
            tma_reduce_add_4d(&a.tm_dq, sbase + dq_box<D>(s, cc) + quarter * 32 * 128, rd * HALF + 32 * cc, h,
                              qt * 128 + (int)quarter * 32, bu.b);
          bulk_commit();
        };
        // round 0: columns [0, HALF) -> the dO_i buffer (dP_i and dV_i, its
        // readers, completed before dQ_i did)
        {
          uint32_t v[HALF];
#pragma unroll
          for (int c = 0; c < HALF; c += 32) RA_TMEM_LD32(T_DP + lane_off + c, (v + c));
          tmem_ld_wait();
          stage(v);
        }
        if (lane == 0) reduce(0);
        // round 1's columns stay in registers; the TMEM columns go back to the MMA warp
        uint32_t v1[HALF];
#pragma unroll
        for (int c = 0; c < HALF; c += 32) RA_TMEM_LD32(T_DP + lane_off + HALF + c, (v1 + c));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(BAR_DQ_FREE);
        if (lane == 0) bulk_wait_read_all();  // this warp's round-0 rows have left shared memory
        __syncwarp();
        // round 1: columns [HALF, D) into the same rows
        stage(v1);
        if (lane == 0) {
          reduce(1);
          bulk_wait_read_all();  // the dO buffer may be refilled once the TMA engine has read it
          mbar_arrive(bar_do_empty(s));
        }
      }
      if (!ok) break;
      if (!mbar_wait(BAR_DKV_FULL, k & 1, abort_flag, a.status, lim)) { ok = false; break; }
      tc_fence_after();
      const long long row = (long long)bu.jt * 128 + r;
      const long long base = lay_at(a.kvl, bu.b, row, bu.g);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t src = (which == 0 ? T_DK : T_DV) + lane_off;
        const float mul = which == 0 ? a.scale : 1.f;
        void* outp = which == 0 ? a.dk : a.dv;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
          RA_TMEM_LD32(src + c, v);
          tmem_ld_wait();
          if (a.grad_dtype == RA_F32) {
            float* op = static_cast<float*>(outp) + base + c;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(op + j) =
                  make_float4(__uint_as_float(v[j]) * mul, __uint_as_float(v[j + 1]) * mul,
                              __uint_as_float(v[j + 2]) * mul, __uint_as_float(v[j + 3]) * mul);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float f0 = __uint_as_float(v[j]) * mul, f1 = __uint_as_float(v[j + 1]) * mul;
              if (a.grad_dtype == RA_BF16) {
                __nv_bfloat162 t = __floats2bfloat162_rn(f0, f1);
                pk[j / 2] = *reinterpret_cast<uint32_t*>(&t);
              } else {
                pk[j / 2] = pack_half2(f0, f1);
              }
            }
            uint4* op = reinterpret_cast<uint4*>(static_cast<uint16_t*>(outp) + base + c);
#pragma unroll
            for (int j = 0; j < 4; ++j) op[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR_DKV_FREE);
      ++k;
    }
    if (lane == 0) bulk_wait_all();  // this warp's reductions complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tc_bwd(TcBwdArgs& a, int num_sms, cudaStream_t st) {
  if (a.num_units <= 0) return cudaSuccess;
  const int grid = a.num_units < num_sms ? a.num_units : num_sms;
  cudaError_t e;
  auto run = [&](auto kernel, int smem) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, smem, st>>>(a);
    return cudaSuccess;
  };
  if (a.d == 128) {
    if (a.striped)
      e = a.precise ? run(tc_bwd_kernel<128, true, kLayoutStriped>, BwdSmem<128>::kBytes)
                    : run(tc_bwd_kernel<128, false, kLayoutStriped>, BwdSmem<128>::kBytes);
    else if (a.host_len)
      e = a.precise ? run(tc_bwd_kernel<128, true, kLayoutVarlen>, BwdSmem<128>::kBytes)
                    : run(tc_bwd_kernel<128, false, kLayoutVarlen>, BwdSmem<128>::kBytes);
    else
      e = a.precise ? run(tc_bwd_kernel<128, true, kLayoutContiguous>, BwdSmem<128>::kBytes)
                    : run(tc_bwd_kernel<128, false, kLayoutContiguous>, BwdSmem<128>::kBytes);
  } else if (a.d == 64) {
    if (a.striped)
      e = a.precise ? run(tc_bwd_kernel<64, true, kLayoutStriped>, BwdSmem<64>::kBytes)
                    : run(tc_bwd_kernel<64, false, kLayoutStriped>, BwdSmem<64>::kBytes);
    else if (a.host_len)
      e = a.precise ? run(tc_bwd_kernel<64, true, kLayoutVarlen>, BwdSmem<64>::kBytes)
                    : run(tc_bwd_kernel<64, false, kLayoutVarlen>, BwdSmem<64>::kBytes);
    else
      e = a.precise ? run(tc_bwd_kernel<64, true, kLayoutContiguous>, BwdSmem<64>::kBytes)
                    : run(tc_bwd_kernel<64, false, kLayoutContiguous>, BwdSmem<64>::kBytes);
  } else {
    return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace ra
