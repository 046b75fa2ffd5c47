// Forward blockwise attention on the sm_103a tensor cores (tcgen05 + TMEM +
// TMA), for the ring of virtual hosts and for a single (Q block, KV block)
// step.
//
// What it computes: for every query row, the online-softmax state over the
// key/value tiles it sees, visited in ring order -- host i takes key/value
// blocks (i - s) mod P, s = 0, 1, ... ("Ring Attention: Train 1M Tokens on
// 8GB GPUs in 2026", section "Ring Attention: Partition Sequence Length, Not
// Batch"), each block's tiles from the last to the first -- merged with the
// rescaled (max, exp_sum, weighted_output) rule of its "Gotchas and Failure
// Modes" section, then normalised (O = o / l, LSE = m + ln l).  Blocks wholly
// in a query tile's causal future are skipped; only tiles that straddle the
// diagonal (or the ragged end of a block) are masked element by element.
//
// CTA organisation (one persistent CTA per SM, 10 warps):
//   warp 0      TMA producer: Q tiles of the unit, then K(0), V(0), K(1), ...
//               through a ring of shared-memory stages
//   warp 1      allocates TMEM; one lane issues every tcgen05.mma
//   warps 2-5   softmax warpgroup for query tile A (thread = row)
//   warps 6-9   softmax warpgroup for query tile B (the next 128 rows)
// A unit is a pair of 128-row query tiles of one (batch, head) in one host,
// so every K/V tile brought into shared memory feeds two tiles of MMAs.
//
// TMEM (512 columns x 128 lanes, fp32): S_A [0,128) S_B [128,256)
// O_A [256, 256+D) O_B [256+D, 256+2D).  The softmax warps overwrite the
// first 64 columns of S_X with P_X as packed fp16 pairs, which the PV MMA
// reads directly from TMEM (A operand), so P never touches shared memory.
// The MMA order per iteration is  PV_A(it) S_A(it+1) PV_B(it) S_B(it+1):
// while one warpgroup computes its softmax the tensor core works on the
// other tile.
//
// Numerics: S = Q K^T accumulates in fp32 from bf16/fp16 operands; scores
// are scaled in the exponent (exp2 with log2(e) folded into the scale);
// P is rounded to fp16 and V is fp16, O accumulates in fp32.  With PRECISE,
// P is carried as two fp16 terms (hi = fp16(p), lo = fp16(p - hi), the lo
// term in S_X columns [64,128)) and both are multiplied by V, which brings
// the rounding of P from 2^-12 relative to about 2^-24.  The running
// maximum is updated lazily: O and l are rescaled only when the maximum
// grows by more than 8 (log2 units), so P <= 2^8, well inside fp16.
#include <math.h>

#include <type_traits>

#include "ra_device.cuh"

namespace ra {
namespace {

constexpr int kThreads = 320;
constexpr int kStages = 4;  // the MMA loop relies on K/V stage pairs (1, 2) and (3, 0)
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row tile, fp16/bf16
  static constexpr int kQA = 0;
  static constexpr int kQB = kTileBytes;
  static constexpr int kStage0 = 2 * kTileBytes;
  static constexpr int kBars = kStage0 + kStages * kTileBytes;
  // barriers: q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2],
  // o_full[2], drain, unit_full[4], unit_empty[4]
  static constexpr int kNumBars = 2 + 2 * kStages + 6 + 1 + 8;
  static constexpr int kMisc = kBars + kNumBars * 8;  // tmem slot, abort flag
  static constexpr int kUnits = kMisc + 16;           // unit ring: 4 unit indices
  static constexpr int kBytes = kUnits + 16;
  // slack for 1024-byte alignment; at least 120 KB so that one CTA (holding
  // all 512 TMEM columns) occupies an SM
  static constexpr int kAlloc = (kBytes + 1024) > 122880 ? (kBytes + 1024) : 122880;
};

struct UnitInfo {
  int b, h, g;
  int qa_row0;    // tensor row of tile A (tile B = qa_row0 + 128)
  int has_b;
  int n_iter;     // key/value tiles visited
  int start[2];   // contiguous layouts: first iteration at which tile A / B is active
  long long qpos0[2];  // global position of row 0 of tile A / B
  // key/value tile at iteration it (contiguous layouts):
  //   kt = ring_noncausal ? (kt0 - it) mod nkt : kt0 - it
  int kt0;
  int nkt;
  int wrap;
  // striped causal ring: host `host` visits blocks (host - s) mod P, and in
  // each block the local tiles lead, lead-1, ..., 0 (L = lead + 1 per block)
  int striped, host, P, T, L, tq[2];
  unsigned long long L_m;  // div_magic(L)
};

__device__ __forceinline__ int host_len_at(const int* hl, int j, int S) {
  const int v = __ldg(hl + j);
  return v < 0 ? 0 : (v > S ? S : v);
}

// Key/value tile of iteration it: global tile kt, and for striped layouts the
// local tile tk and the block j it belongs to.
__device__ __forceinline__ int kt_at(const UnitInfo& u, int it, int* tk = nullptr, int* blk = nullptr) {
  if (u.striped) {
    const int s = div_by(it, u.L_m);
    const int t = u.kt0 - (it - s * u.L);
    int j = u.host - s;
    if (j < 0) j += u.P;
    if (tk) *tk = t;
    if (blk) *blk = j;
    return j * u.T + t;
  }
  int kt = u.kt0 - it;
  if (u.wrap && kt < 0) kt += u.nkt;
  return kt;
}

// With variable host lengths a key/value tile wholly in a host's padding is
// skipped by every role.
// Valid keys in the key/value tile of iteration it (<= 0: wholly padding).
__device__ __forceinline__ int kv_tile_len(const UnitInfo& u, int it, const TcFwdArgs& a) {
  int kt = u.kt0 - it;  // contiguous ring tiles
  if (u.wrap && kt < 0) kt += u.nkt;
  const int T = a.ring_S / 128;
  const int j = div_by(kt, a.T_m), tk = kt - j * T;
  return host_len_at(a.host_len, j, a.ring_S) - tk * 128;
}
__device__ __forceinline__ bool iter_valid(const UnitInfo& u, int it, const TcFwdArgs& a) {
  return kv_tile_len(u, it, a) > 0;
}
__device__ __forceinline__ int next_valid(const UnitInfo& u, int it, const TcFwdArgs& a) {
  ++it;
  while (it < u.n_iter && !iter_valid(u, it, a)) ++it;
  return it;
}

// Does query tile x (0 = A, 1 = B) take part in iteration it?
__device__ __forceinline__ bool active(const UnitInfo& u, int x, int it) {
  if (u.striped) {
    if (x == 1) return u.has_b;
    return u.kt0 - (it - div_by(it, u.L_m) * u.L) <= u.tq[0];
  }
  return it >= u.start[x];
}

__device__ __forceinline__ bool ever_active(const UnitInfo& u, int x) {
  return u.striped ? (x == 0 || u.has_b) : u.start[x] < u.n_iter;
}

// Last key/value tile with at least one key visible to some row of a query
// tile whose first row is at position qpos0 and last valid row at qpos_last.
__device__ __forceinline__ int last_visible_tile(const TcFwdArgs& a, long long qpos_last,
                                                 int nkt) {
  if (!a.causal) return nkt - 1;
  const long long lim = qpos_last - a.kv_off;  // keys at row index <= lim are visible
  if (lim < 0) return -1;
  const long long t = lim / 128;
  return (int)(t < nkt - 1 ? t : nkt - 1);
}

// Units are ordered head-major (all resident CTAs sweep the key/value tiles
// of one (batch, head) together, which keeps them in L2), and within a head
// from the last query tiles to the first: under a causal mask the last ones
// see the most keys.  The ring forward's CTAs draw units in this order from
// a counter in global memory, so none runs ahead into another head and the
// lightest units end the launch.
// VARLEN selects the kernel built for variable host lengths; the other
// builds see no length array and compile its checks away.
template <bool VARLEN, bool STRIPED>
__device__ __forceinline__ UnitInfo unit_info(const TcFwdArgs& a, int u) {
  UnitInfo r;
  int per_head;
  if (a.ring_P > 0) {
    const int T = a.ring_S / 128;
    per_head = a.ring_P * ((T + 1) / 2);
  } else {
    per_head = (((a.Nq + 127) / 128) + 1) / 2;
  }
  const int bh = u / per_head;
  const int pidx_desc = u % per_head;
  r.b = bh / a.Hq;
  r.h = bh % a.Hq;
  r.g = r.h / (a.Hq / a.Hkv);
  const int nkt = (a.Nkv + 127) / 128;
  r.nkt = nkt;
  r.striped = 0;
  if (STRIPED) {
    // striped: the row of a host's local row l holds position l * P + host; every
    // host has the same work, heaviest local pairs first
    const int T = a.ring_S / 128;
    const int pph = (T + 1) / 2;
    const int lp = pph - 1 - pidx_desc / a.ring_P;
    const int host = pidx_desc % a.ring_P;
    r.qa_row0 = host * a.ring_S + lp * 256;
    r.has_b = (2 * lp + 1) < T;
    r.qpos0[0] = r.qa_row0;  // unused for striped masks
    r.qpos0[1] = r.qa_row0 + 128;
    r.striped = 1;
    r.host = host;
    r.P = a.ring_P;
    r.T = T;
    r.tq[0] = 2 * lp;
    r.tq[1] = 2 * lp + 1;
    r.kt0 = r.has_b ? r.tq[1] : r.tq[0];  // lead local tile
    r.L = r.kt0 + 1;
    r.L_m = div_magic((unsigned)r.L);
    r.n_iter = a.ring_P * r.L;
    r.wrap = 0;
    r.start[0] = r.start[1] = 0;
    return r;
  }
  if (a.ring_P > 0) {
    const int T = a.ring_S / 128;
    const int pph = (T + 1) / 2;
    const int total = a.ring_P * pph;
    const int pg = total - 1 - pidx_desc;  // heaviest (latest) pairs first
    const int host = pg / pph, lp = pg % pph;
    r.qa_row0 = host * a.ring_S + lp * 256;
    r.has_b = (2 * lp + 1) < T;
    const int ta = r.qa_row0 / 128;
    const int lead = r.has_b ? ta + 1 : ta;
    r.qpos0[0] = r.qa_row0;
    r.qpos0[1] = r.qa_row0 + 128;
    if (a.causal) {
      r.kt0 = lead;
      r.n_iter = lead + 1;
      r.wrap = 0;
      r.start[0] = lead - ta;
      r.start[1] = 0;
    } else {
      r.kt0 = (host + 1) * T - 1;
      r.n_iter = nkt;
      r.wrap = 1;
      r.start[0] = 0;
      r.start[1] = 0;
    }
    if (VARLEN && a.host_len) {
      // query tiles wholly in the host's padding do no work (their rows were
      // filled with O = 0, LSE = -inf beforehand)
      const int qlen = host_len_at(a.host_len, host, a.ring_S);
      const int la = lp * 256;
      if (la >= qlen) {
        r.n_iter = 0;  // both tiles padding: the whole unit is skipped
      } else if (la + 128 >= qlen && r.has_b) {
        r.has_b = 0;
        r.start[1] = r.n_iter;
        if (a.causal) {  // tile A leads
          r.kt0 = ta;
          r.n_iter = ta + 1;
          r.start[0] = 0;
          r.start[1] = r.n_iter;
        }
      }
    }
  } else {
    const int nqt = (a.Nq + 127) / 128;
    const int total = (nqt + 1) / 2;
    const int lp = total - 1 - pidx_desc;
    r.qa_row0 = lp * 256;
    r.has_b = (r.qa_row0 + 128) < a.Nq;
    r.qpos0[0] = a.q_off + r.qa_row0;
    r.qpos0[1] = a.q_off + r.qa_row0 + 128;
    const long long lastA = a.q_off + min(r.qa_row0 + 127, a.Nq - 1);
    const int ktA = last_visible_tile(a, lastA, nkt);
    int ktB = -1;
    if (r.has_b) ktB = last_visible_tile(a, a.q_off + min(r.qa_row0 + 255, a.Nq - 1), nkt);
    const int lead = r.has_b ? max(ktA, ktB) : ktA;
    r.kt0 = lead;
    r.n_iter = lead + 1;
    r.wrap = 0;
    r.start[0] = ktA >= 0 ? lead - ktA : r.n_iter;      // never active if no key visible
    r.start[1] = r.has_b ? (ktB >= 0 ? lead - ktB : r.n_iter) : r.n_iter;
  }
  if (!r.has_b) r.start[1] = r.n_iter;
  return r;
}

template <int D, bool PRECISE, bool VARLEN, bool STRIPED>
__global__ void __launch_bounds__(kThreads, 1) tc_fwd_kernel(const __grid_constant__ TcFwdArgs a) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBars;
  const uint32_t BAR_Q_FULL = bar0, BAR_Q_EMPTY = bar0 + 8;
  auto bar_kv_full = [&](int s) { return bar0 + 16 + 8 * s; };
  auto bar_kv_empty = [&](int s) { return bar0 + 16 + 8 * kStages + 8 * s; };
  const uint32_t bar_x = bar0 + 16 + 16 * kStages;
  auto bar_s_full = [&](int x) { return bar_x + 8 * x; };
  auto bar_p_full = [&](int x) { return bar_x + 16 + 8 * x; };
  auto bar_o_full = [&](int x) { return bar_x + 32 + 8 * x; };
  const uint32_t BAR_DRAIN = bar_x + 48;
  auto bar_unit_full = [&](int s) { return bar_x + 56 + 8 * s; };
  auto bar_unit_empty = [&](int s) { return bar_x + 88 + 8 * s; };
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + L::kUnits);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(BAR_Q_FULL, 1);
    mbar_init(BAR_Q_EMPTY, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar_s_full(x), 1);
      mbar_init(bar_p_full(x), 128);
      mbar_init(bar_o_full(x), 1);
    }
    mbar_init(BAR_DRAIN, 1);
    // the producer draws the CTA's units and passes them on through a ring of
    // four slots; every consumer thread (MMA lane, 256 softmax threads) hands
    // a slot back once it has read it
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar_unit_full(s), 1);
      mbar_init(bar_unit_empty(s), 1 + 256);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t lim = a.wait_limit_ns;
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
      const uint64_t pol_kv = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      uint32_t L_cnt = 0;  // K/V loads issued
      int k = 0;
      bool ok = true;
      uint32_t last_phase[kStages];
      int issued[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = 0, last_phase[s] = 0;
      int q_issued = 0;
      // n counts the units this CTA has drawn; a draw at or past the last
      // unit ends every role
      for (int n = 0; ok; ++n) {
        const int slot = n & 3;
        if (!mbar_wait(bar_unit_empty(slot), ((n >> 2) & 1) ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
        const int u = a.sched ? (int)atomicAdd(a.sched, 1u) : (int)blockIdx.x + n * (int)gridDim.x;
        unit_ring[slot] = u;
        mbar_arrive(bar_unit_full(slot));
        if (u >= a.num_units) break;
        const UnitInfo ui = unit_info<VARLEN, STRIPED>(a, u);
        if (ui.n_iter == 0) continue;  // no key of this block is visible to the unit
        if (!mbar_wait(BAR_Q_EMPTY, (k & 1) ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
        ++k;
        const uint32_t qbytes = (ui.has_b ? 2 : 1) * L::kTileBytes;
        mbar_arrive_expect_tx(BAR_Q_FULL, qbytes);
        q_issued = 1;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sbase + L::kQA + c * 16384, &a.tm_q, BAR_Q_FULL, c * 64, ui.h,
                      ui.qa_row0, ui.b, pol_q);
          if (ui.has_b)
            tma_load_4d(sbase + L::kQB + c * 16384, &a.tm_q, BAR_Q_FULL, c * 64, ui.h,
                        ui.qa_row0 + 128, ui.b, pol_q);
        }
        for (int it = 0; it < ui.n_iter && ok; ++it) {
          if (VARLEN && !iter_valid(ui, it, a)) continue;
          int tk = 0, blk = 0;
          const int kt = kt_at(ui, it, &tk, &blk);
          if (a.log.entries) log_visit(a.log, 0u, ui.b * a.Hq + ui.h, ui.qa_row0 / 128, kt);
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {  // K then V
            const int s = L_cnt % kStages;
            const uint32_t ph = (L_cnt / kStages) & 1;
            if (!mbar_wait(bar_kv_empty(s), ph ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
            mbar_arrive_expect_tx(bar_kv_full(s), L::kTileBytes);
            const CUtensorMap* tm = kv == 0 ? &a.tm_k : &a.tm_v;
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_4d(sbase + L::kStage0 + s * L::kTileBytes + c * 16384, tm,
                          bar_kv_full(s), c * 64, ui.g, kt * 128, ui.b, pol_kv);
            issued[s] = 1;
            last_phase[s] = ph;
            ++L_cnt;
          }
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA exits
        const uint64_t drain = 100000000ull;
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) (void)mbar_wait(bar_kv_full(s), last_phase[s], abort_flag, nullptr, drain);
        if (q_issued) (void)mbar_wait(BAR_Q_FULL, (k - 1) & 1, abort_flag, nullptr, drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_f16(a.qk_bf16 ? 1u : 0u, 0, 0, 128, 128);
      const uint32_t idesc_pv = idesc_f16(0, 0, 1, 128, D);
      const uint32_t tS[2] = {tmem + 0u, tmem + 128u};
      const uint32_t tO[2] = {tmem + 256u, tmem + 256u + (uint32_t)D};
      uint32_t L_cnt = 0;
      uint32_t p_cnt[2] = {0, 0};
      int k = 0;
      bool ok = true;
      // descriptors built once; each MMA advances one with a single add
      const uint64_t dQ_k[2] = {smem_desc_sw128(sbase + L::kQA, 16, 1024), smem_desc_sw128(sbase + L::kQB, 16, 1024)};
      const uint64_t dKV_k0 = smem_desc_sw128(sbase + L::kStage0, 16, 1024);
      const uint64_t dKV_mn0 = smem_desc_sw128(sbase + L::kStage0, 16384, 1024);
      constexpr uint32_t kStageStep = L::kTileBytes >> 4;
      auto issue_s = [&](int x, uint32_t kstage) {
        const uint64_t da = dQ_k[x], db = dKV_k0 + kstage * kStageStep;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tS[x], desc_off(da, off), desc_off(db, off), idesc_qk, kk > 0);
        }
        mma_commit(bar_s_full(x));
      };
      auto issue_pv = [&](int x, uint32_t vstage, bool accumulate) {
        const uint64_t db = dKV_mn0 + vstage * kStageStep;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_ts(tO[x], tS[x] + kk * 8, desc_off(db, kk * 2048), idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
        }
        if (PRECISE) {  // + P_lo V
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ts(tO[x], tS[x] + 64 + kk * 8, desc_off(db, kk * 2048), idesc_pv, 1u);
        }
      };
      for (int n = 0; ok; ++n) {
        int u;
        if (!take_unit(n, &u) || u >= a.num_units) break;
        const UnitInfo ui = unit_info<VARLEN, STRIPED>(a, u);
        if (ui.n_iter == 0) continue;
        if (!mbar_wait(BAR_Q_FULL, k & 1, abort_flag, a.status, lim)) { ok = false; break; }
        ++k;
        tc_fence_after();
        // prologue: S of the first valid iteration
        const int it0 = !VARLEN || iter_valid(ui, 0, a) ? 0 : next_valid(ui, 0, a);
        uint32_t sk = L_cnt % kStages;
        if (!mbar_wait(bar_kv_full(sk), (L_cnt / kStages) & 1, abort_flag, a.status, lim)) { ok = false; break; }
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (active(ui, x, it0)) issue_s(x, sk);
        mma_commit(bar_kv_empty(sk));
        ++L_cnt;
        bool first_pv[2] = {a.mode == 0, a.mode == 0};
        // A unit takes an even number of K/V loads (its first K, then V(it)
        // and K(it+1) per iteration, V alone at the last), so V(it) sits in
        // stage 1 or 3 and K(it+1) in the stage after it, alternating from one
        // iteration to the next.  Each iteration is built for its stage pair,
        // which makes the descriptors and barrier addresses constants: with
        // stage numbers computed at run time the descriptor arithmetic held the
        // issue of each MMA above the tensor pipe's 64 cycles.
        static_assert(kStages == 4, "stage pairs (1, 2) and (3, 0)");
        int it = it0;
        auto step = [&](auto sv_c) {  // false once the unit is done or a wait gave up
          constexpr uint32_t sv = decltype(sv_c)::value, sk2 = (sv + 1) % kStages;
          const int nx = VARLEN ? next_valid(ui, it, a) : it + 1;
          if (!mbar_wait(bar_kv_full(sv), (L_cnt / kStages) & 1, abort_flag, a.status, lim)) return ok = false;
          ++L_cnt;
          const bool has_next = nx < ui.n_iter;
          if (has_next) {
            if (!mbar_wait(bar_kv_full(sk2), (L_cnt / kStages) & 1, abort_flag, a.status, lim)) return ok = false;
            ++L_cnt;
          }
          tc_fence_after();
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (active(ui, x, it)) {
              if (!mbar_wait(bar_p_full(x), p_cnt[x] & 1, abort_flag, a.status, lim)) return ok = false;
              ++p_cnt[x];
              tc_fence_after();
              issue_pv(x, sv, !first_pv[x]);
              first_pv[x] = false;
              if (!has_next) mma_commit(bar_o_full(x));
            }
            if (has_next && active(ui, x, nx)) issue_s(x, sk2);
          }
          mma_commit(bar_kv_empty(sv));
          if (has_next) mma_commit(bar_kv_empty(sk2));
          it = nx;
          return it < ui.n_iter;
        };
        bool more = it < ui.n_iter;
        if (more && L_cnt % kStages == 3) more = step(std::integral_constant<uint32_t, 3>{});
        while (more) {
          more = step(std::integral_constant<uint32_t, 1>{});
          if (more) more = step(std::integral_constant<uint32_t, 3>{});
        }
        if (!ok) break;
        mma_commit(BAR_Q_EMPTY);
      }
      // wait for every MMA issued to finish before TMEM is released
      mma_commit(BAR_DRAIN);
      (void)mbar_wait(BAR_DRAIN, 0, abort_flag, nullptr, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 2) / 4;                 // 0: tile A, 1: tile B
    const uint32_t quarter = warp & 3;            // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;            // row within the tile
    const uint32_t lane_off = (quarter * 32) << 16;
    const uint32_t tS = tmem + (x == 0 ? 0u : 128u) + lane_off;
    const uint32_t tO = tmem + 256u + (x == 0 ? 0u : (uint32_t)D) + lane_off;
    const float sl2 = a.scale_log2;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      int u;
      if (!take_unit(n, &u) || u >= a.num_units) break;
      const UnitInfo ui = unit_info<VARLEN, STRIPED>(a, u);
      if ((VARLEN && ui.n_iter == 0) || !ever_active(ui, x)) continue;  // this tile sees no key in this unit
      const int row = ui.qa_row0 + x * 128 + r;  // tensor row
      // with variable host lengths, rows past their host's valid length are padding
      const bool row_ok = row < a.Nq && (!VARLEN || row % a.ring_S < host_len_at(a.host_len, row / a.ring_S, a.ring_S));
      const long long qpos = ui.qpos0[x] + r;
      float m_run = -INFINITY, l_run = 0.f;
      // row offsets of the state (m, l: [B, Hq, N]; o: [B, N, Hq, D]), formed where used
      auto sidx = [&]() { return ((long long)ui.b * a.Hq + ui.h) * a.Nq + row; };
      auto oidx = [&]() { return (((long long)ui.b * a.Nq + row) * a.Hq + ui.h) * D; };
      if (a.mode == 1) {
        // load the running state into registers and TMEM
        if (row_ok) {
          const float mm = a.m_acc[sidx()];
          m_run = mm == -INFINITY ? -INFINITY : mm * kLog2e;
          l_run = a.l_acc[sidx()];
        }
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 f = row_ok ? *reinterpret_cast<const float4*>(a.o_acc + oidx() + c + j)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            v[j] = __float_as_uint(f.x);
            v[j + 1] = __float_as_uint(f.y);
            v[j + 2] = __float_as_uint(f.z);
            v[j + 3] = __float_as_uint(f.w);
          }
          RA_TMEM_ST32(tO + c, v);
        }
      }
      bool o_valid = (a.mode == 1);  // O_X holds a state that must be rescaled
      for (int it = ui.striped ? 0 : ui.start[x]; it < ui.n_iter; ++it) {
        if (!active(ui, x, it)) continue;
        int kv_len = 128;  // valid keys of this tile (variable host lengths)
        if (VARLEN) {
          kv_len = kv_tile_len(ui, it, a);
          if (kv_len <= 0) continue;
        }
        if (!mbar_wait(bar_s_full(x), s_cnt & 1, abort_flag, a.status, lim)) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        int tk = 0, blk = 0;
        const int kt = kt_at(ui, it, &tk, &blk);
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 128; c += 32) RA_TMEM_LD32(tS + c, (sr + c));
        tmem_ld_wait();
        // element masks: causal diagonal tiles and the ragged end of the keys
        const long long kvpos0 = a.kv_off + (long long)kt * 128;
        bool need_mask;
        long long lim_c;  // column c of the tile is visible iff c <= lim_c
        if (ui.striped) {
          // same local tile: key row c sees query row r iff c < r, or c == r and
          // the key's host is not after the query's
          need_mask = tk == ui.tq[x];
          lim_c = r - (blk > ui.host ? 1 : 0);
        } else {
          need_mask = (a.causal && kvpos0 + 127 > ui.qpos0[x]) || (kt * 128 + 128 > a.Nkv);
          lim_c = a.causal ? qpos - kvpos0 : 127;
        }
        if (VARLEN && kv_len < 128) need_mask = true;  // keys past the host's valid length
        if (need_mask) {
          const int nvalid = VARLEN ? min(a.Nkv - kt * 128, kv_len) : a.Nkv - kt * 128;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim_c || c >= nvalid) sr[c] = __float_as_uint(-INFINITY);
        }
        // row maximum as eight independent chains of three-input maxima, so
        // the exponentials can start after ~10 dependent steps instead of 127
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mk[k] = fmax3(__uint_as_float(sr[k]), __uint_as_float(sr[k + 8]), __uint_as_float(sr[k + 16]));
#pragma unroll
        for (int c = 24; c < 120; c += 16) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mk[k] = fmax3(mk[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], __uint_as_float(sr[120 + k]));
        const float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
        const float m_tile = mx * sl2;  // -inf stays -inf (scale > 0)
        float m_use = m_run;
        if (m_tile > m_run + kRescaleThreshold) m_use = m_tile;  // also when m_run = -inf
        const bool rescale = (m_use != m_run);
        const float alpha = rescale ? ex2_approx(m_run - m_use) : 1.f;  // exp2(-inf) = 0
        const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use;
        const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
        float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t pk[16];
          uint32_t pl[PRECISE ? 16 : 1];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 e = __ffma2_rn(make_float2(__uint_as_float(sr[c + j]), __uint_as_float(sr[c + j + 1])),
                                        sl2x2, nm2);
            const float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
            rs2[(j / 2) & 1] = __fadd2_rn(rs2[(j / 2) & 1], make_float2(p0, p1));
            pk[j / 2] = pack_half2(p0, p1);
            if (PRECISE) {
              const float2 hi = unpack_half2(pk[j / 2]);
              pl[j / 2] = pack_half2(p0 - hi.x, p1 - hi.y);
            }
          }
          RA_TMEM_ST16(tS + c / 2, pk);
          if (PRECISE) RA_TMEM_ST16(tS + 64 + c / 2, pl);
        }
        const float rs = (rs2[0].x + rs2[1].x) + (rs2[0].y + rs2[1].y);
        l_run = l_run * alpha + rs;
        m_run = m_use;
        if (o_valid && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            RA_TMEM_LD32(tO + c, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            RA_TMEM_ST32(tO + c, ov);
          }
        }
        o_valid = true;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p_full(x));
      }
      if (!ok) break;
      if (!mbar_wait(bar_o_full(x), o_cnt & 1, abort_flag, a.status, lim)) { ok = false; break; }
      ++o_cnt;
      tc_fence_after();
      // epilogue
      if (a.mode == 0) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const long long out = lay_at(a.ol, ui.b, row, ui.h);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          RA_TMEM_LD32(tO + c, ov);
          tmem_ld_wait();
          if (row_ok) {
            if (a.o_dtype == RA_F32) {
              float* op = static_cast<float*>(a.o_out) + out + c;
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(op + j) =
                    make_float4(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv,
                                __uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
            } else {
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float f0 = __uint_as_float(ov[j]) * inv, f1 = __uint_as_float(ov[j + 1]) * inv;
                if (a.o_dtype == RA_BF16) {
                  __nv_bfloat162 t = __floats2bfloat162_rn(f0, f1);
                  pk[j / 2] = *reinterpret_cast<uint32_t*>(&t);
                } else {
                  pk[j / 2] = pack_half2(f0, f1);
                }
              }
              uint4* op = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o_out) + out + c);
#pragma unroll
              for (int j = 0; j < 4; ++j) op[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
          }
        }
        if (row_ok) a.lse[sidx()] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      } else {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          RA_TMEM_LD32(tO + c, ov);
          tmem_ld_wait();
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(a.o_acc + oidx() + c + j) =
                  make_float4(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1]),
                              __uint_as_float(ov[j + 2]), __uint_as_float(ov[j + 3]));
          }
        }
        if (row_ok) {
          a.m_acc[sidx()] = m_run == -INFINITY ? -INFINITY : m_run * kLn2;
          a.l_acc[sidx()] = l_run;
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tc_fwd(TcFwdArgs& a, int num_sms, cudaStream_t st) {
  if (a.num_units <= 0) return cudaSuccess;
  const int grid = a.num_units < num_sms ? a.num_units : num_sms;
  cudaError_t e;
  auto run = [&](auto kernel, int smem) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, smem, st>>>(a);
    return cudaSuccess;
  };
  // variable host lengths and the striped layout never come together (the
  // entry points reject the pair)
  auto pick = [&](auto d_c) {
    constexpr int DD = decltype(d_c)::value;
    constexpr int smem = FwdSmem<DD>::kAlloc;
    const bool striped = a.ring_P > 0 && a.striped;
    if (a.host_len)
      return a.precise ? run(tc_fwd_kernel<DD, true, true, false>, smem) : run(tc_fwd_kernel<DD, false, true, false>, smem);
    if (striped)
      return a.precise ? run(tc_fwd_kernel<DD, true, false, true>, smem) : run(tc_fwd_kernel<DD, false, false, true>, smem);
    return a.precise ? run(tc_fwd_kernel<DD, true, false, false>, smem) : run(tc_fwd_kernel<DD, false, false, false>, smem);
  };
  if (a.d == 128)
    e = pick(std::integral_constant<int, 128>{});
  else if (a.d == 64)
    e = pick(std::integral_constant<int, 64>{});
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace ra
