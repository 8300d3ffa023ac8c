// mha_fwd_wide.cu -- bf16 attention forward for heads wider than 128
// features (d_k and d_v up to 256) on the 5th-generation tensor cores, sm_103a.
//
// The same operation as mha_fwd_bf16.cu,
//   O = softmax(Q K^T * scale) V
// ("Attention Is All You Need", Section 3.2.1, Equation (1): keys of
// dimension d_k, values of dimension d_v, any width), with the online
// softmax of that file (a per-row reference maximum moved only when a tile's
// maximum exceeds it by more than 8 in log2 units; shift invariance, formula
// page transformer-attention, section 証明).  A 256-wide head does not fit
// that kernel's tiling: two 128-row output tiles of 256 float32 columns alone
// fill the 512 TMEM columns.  Here a unit is one 128-row query tile of one
// (b, h), and TMEM holds
//   O (256 columns) | Q (128 columns: 256 bf16 features in pairs) | S0 | S1
// with S0, S1 two 64-column score buffers (64-key tiles) and the weights P of
// a tile written as bf16 pairs over the first 32 columns of its own buffer.
// Q sits in TMEM as the A operand of S = Q K^T, so both products read only
// K or V from shared memory (S: 2 KB per K16 step, P.V: 8 KB per 128-cycle
// step): 4 KB of K and V per 64 cycles of tensor work plus the same again
// written by TMA, the 128 B/clk shared-memory rate.  Per 64-key tile the
// tensor core does 1024 cycles of work and the softmax (64 scores per row,
// one row per thread) about half of that, so one softmax warpgroup keeps up.
//
// 256 threads in four roles:
//   warps 0-3  softmax + epilogue (thread r owns query row r = TMEM lane r);
//              right after a unit's last weights (before its epilogue) they
//              copy the next unit's Q tile from shared memory into TMEM (one
//              row each), so the next unit's first scores are computed while
//              the epilogue runs
//   warp 4     TMEM allocator and MMA issuer: S(0), S(1), PV(0), S(2), PV(1),
//              ..., so S(j+1) runs while the softmax works on S(j), and S(j+2)
//              overwrites P(j) only after PV(j) read it (MMAs of one thread
//              run in order)
//   warp 5     TMA producer: the next unit's Q into a staging buffer, then K_j
//              and V_j (64 keys x 256 features) into two-stage rings
//   warp 6     scheduler: the grid has one CTA per unit, but CTAs are
//              persistent: once a CTA runs, this warp cancels CTAs that have
//              not started (cluster launch control) and feeds their units to
//              the other roles through a two-slot queue, so the hardware's
//              launch order balances the work dynamically (a static striding
//              of the causal units left the busiest SM 24 % above the mean)
//   warp 7     idle
// Units are ordered in groups of heads whose K/V stay in L2, heaviest causal
// query tiles first.
// Causal key tiles past a query tile's last row are never loaded; the
// diagonal tiles and a ragged last tile are masked per element.  Every wait
// is bounded (abort flag, MHA_ERR_TIMEOUT in the status word).
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

constexpr int kWThreads = 256;
constexpr int kWMmaWarp = 4, kWProducerWarp = 5, kWSchedulerWarp = 6;
constexpr int kWConsumers = 6;    // unit-queue readers: 4 softmax warps, the MMA and producer warps
constexpr int kWKeys = 64;        // keys per K / V tile
constexpr int kWStages = 2;       // K and V ring stages
constexpr float kWRescaleThreshold = 8.0f;
constexpr long long kWHeadGroupBytes = 32ll << 20;
constexpr int kRoleWProducer = 11, kRoleWMma = 12, kRoleWSoftmax = 13, kRoleWScheduler = 14;

// W: the widest head the instantiation takes (256, or 64 for the light
// variant whose CTAs fit two to an SM)
template <int W>
struct WCfg {
  static constexpr int NCH = W / 64;                   // 64-feature chunks
  static constexpr int Q_CHUNK = 128 * 128;            // [128 rows x 128 B]
  static constexpr int Q_BYTES = NCH * Q_CHUNK;
  static constexpr int KV_CHUNK = kWKeys * 128;        // [64 keys x 128 B]
  static constexpr int KV_BYTES = NCH * KV_CHUNK;
  static constexpr int OUT_CHUNK = 32 * 128;           // one warp's 32 rows x 64 bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + kWStages * KV_BYTES;
  static constexpr int OFF_OUT = OFF_V + kWStages * KV_BYTES;  // 4 warps x 2 buffers
  static constexpr int OFF_BAR = OFF_OUT + 8 * OUT_CHUNK;
  // barriers
  static constexpr int Q_FULL = 0;        // Q tile staged (TMA)
  static constexpr int Q_STAGE_FREE = 1;  // the softmax copied it to TMEM (128 arrivals)
  static constexpr int Q_TMEM_FULL = 2;   // Q in TMEM (128 arrivals)
  static constexpr int Q_TMEM_FREE = 3;   // the unit's last S is done (TMEM Q reusable)
  static constexpr int S_FULL = 4;        // + buffer
  static constexpr int P_FULL = 6;        // + buffer (128 arrivals)
  static constexpr int PV_DONE = 8;       // each P.V product done
  static constexpr int O_DONE = 9;        // the unit's last P.V done
  static constexpr int O_FREE = 10;       // the epilogue read O (128 arrivals)
  static constexpr int DRAIN = 11;
  static constexpr int K_FULL = 12;
  static constexpr int K_EMPTY = 12 + kWStages;
  static constexpr int V_FULL = 12 + 2 * kWStages;
  static constexpr int V_EMPTY = 12 + 3 * kWStages;
  static constexpr int UNIT_FULL = 12 + 4 * kWStages;   // + slot: unit published
  static constexpr int UNIT_EMPTY = 14 + 4 * kWStages;  // + slot: every consumer read it
  static constexpr int CLC = 16 + 4 * kWStages;         // cancellation response landed
  static constexpr int NBAR = 17 + 4 * kWStages;
  // TMEM slot (+0), abort flag (+4), unit queue (+8, +12), CLC response (+16, 16 bytes)
  static constexpr int OFF_MISC = (OFF_BAR + 8 * NBAR + 15) / 16 * 16;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;
  // TMEM: O (W columns) | Q (W / 2: bf16 pairs) | S0 | S1 (64 each)
  static constexpr uint32_t TM_O = 0, TM_Q = W, TM_S0 = W + W / 2, TM_S1 = TM_S0 + 64;
  static constexpr uint32_t TMEM_COLS = W == 256 ? 512 : 256;
  static_assert(TM_S1 + 64 <= TMEM_COLS, "TMEM budget");
  // CTAs per SM the launch bounds allow
  static constexpr int MIN_BLOCKS = W == 256 ? 1 : 2;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_OUT % 1024 == 0 && OFF_BAR % 8 == 0,
                "alignment");
};

struct WUnit {
  int b, h, q0;  // sequence, head, first query row
  int n;         // key tiles (64 keys each) the query tile sees
  int kv_len;    // keys visible before the causal limit
};

__device__ __forceinline__ WUnit wide_unit(const Bf16Params& p, int u) {
  const int bh_count = p.B * p.H;
  const int nq = p.n_qtiles;
  const int hg = p.head_group;
  const int group = u / (hg * nq);
  const int within = u - group * hg * nq;
  const int heads_here = min(hg, bh_count - group * hg);
  const int tidx = within / heads_here;
  const int bh = group * hg + within % heads_here;
  const int qt = masks_causal(p.mask_kind) ? (nq - 1 - tidx) : tidx;
  WUnit w;
  w.b = bh / p.H;
  w.h = bh % p.H;
  w.q0 = qt * kBlockM;
  int kv_len = p.Lk;
  if (masks_padding(p.mask_kind)) {
    const int len = __ldg(p.key_lens + w.b);
    kv_len = len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
  }
  w.kv_len = kv_len;
  int n = (kv_len + kWKeys - 1) / kWKeys;
  // causal: rows q0 .. q0 + 127 see keys up to q0 + 127
  if (masks_causal(p.mask_kind)) n = min(n, (w.q0 + kBlockM - 1) / kWKeys + 1);
  w.n = n;
  return w;
}

template <int W>
__global__ void __launch_bounds__(kWThreads, WCfg<W>::MIN_BLOCKS)
    fwd_wide_kernel(const __grid_constant__ Bf16Params p) {
  using C = WCfg<W>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::OFF_Q, sK = s_base + C::OFF_K, sV = s_base + C::OFF_V;
  const uint32_t sOut = s_base + C::OFF_OUT;
  auto bar = [&](int id) { return s_base + C::OFF_BAR + 8u * static_cast<uint32_t>(id); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  const uint32_t clc_resp = s_base + C::OFF_MISC + 16;
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  constexpr int S = kWStages;
  // The k-th unit of this CTA from the queue (every consumer warp takes every
  // unit, in order); -1 at the end of the work or when the CTA gave up.
  auto next_unit = [&](int k, int role) {
    const int slot = k & 1;
    if (!mbar_wait(bar(C::UNIT_FULL + slot), (k >> 1) & 1, abort_flag, p.status,
                   role * 64 + C::UNIT_FULL + slot))
      return -1;
    const int u = unit_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C::UNIT_EMPTY + slot));
    return u;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(C::Q_FULL), 1);
    mbar_init(bar(C::Q_STAGE_FREE), 128);
    mbar_init(bar(C::Q_TMEM_FULL), 128);
    mbar_init(bar(C::Q_TMEM_FREE), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::S_FULL + i), 1);
      mbar_init(bar(C::P_FULL + i), 128);
    }
    mbar_init(bar(C::PV_DONE), 1);
    mbar_init(bar(C::O_DONE), 1);
    mbar_init(bar(C::O_FREE), 128);
    mbar_init(bar(C::DRAIN), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(C::K_FULL + s), 1);
      mbar_init(bar(C::K_EMPTY + s), 1);
      mbar_init(bar(C::V_FULL + s), 1);
      mbar_init(bar(C::V_EMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::UNIT_FULL + i), 1);
      mbar_init(bar(C::UNIT_EMPTY + i), kWConsumers);
    }
    mbar_init(bar(C::CLC), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWProducerWarp && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_o);
  }
  if (warp == kWMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if constexpr (W == 64) {
    // A light grid that runs in one wave (two CTAs per SM) lets the next
    // launch on the stream start its set-up in the free slots at once; that
    // launch still waits for this grid before it touches global memory.
    // (Measured, 32 x 8 heads at L 128: -4 %; a persistent grid of more units
    // than slots was 1 % slower with the trigger, so it does not trigger.)
    // (%nsmid counts SM identifiers: at least the SMs, so the test may let a
    // grid slightly larger than one wave trigger, which costs about 1 %)
    uint32_t nsm;
    asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
    if (gridDim.x <= 2 * nsm) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  griddep_wait();  // global memory only from here on

  if (warp == kWProducerWarp) {
    // ---- TMA producer
    const int site = kRoleWProducer * 64;
    int q_cnt = 0, t = 0;  // Q loads, K/V tiles so far
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = next_unit(k, kRoleWProducer);
      if (u < 0) break;
      const WUnit w = wide_unit(p, u);
      if (w.n == 0) continue;
      // the softmax must have copied the previous unit's Q out of the staging buffer
      if (q_cnt > 0 && !mbar_wait(bar(C::Q_STAGE_FREE), (q_cnt - 1) & 1, abort_flag, p.status,
                                  site + C::Q_STAGE_FREE)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(C::Q_FULL), C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sQ + c * C::Q_CHUNK, &p.tm_q, bar(C::Q_FULL), 64 * c, w.h, w.q0, w.b);
      }
      __syncwarp();
      ++q_cnt;
      for (int j = 0; j < w.n; ++j, ++t) {
        const int s = t % S;
        if (t >= S && !mbar_wait(bar(C::K_EMPTY + s), ((t / S) - 1) & 1, abort_flag, p.status,
                                 site + C::K_EMPTY + s)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::K_FULL + s), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(sK + s * C::KV_BYTES + c * C::KV_CHUNK, &p.tm_k, bar(C::K_FULL + s), 64 * c,
                        w.h, j * kWKeys, w.b);
        }
        __syncwarp();
        ++k_issued;
        if (t >= S && !mbar_wait(bar(C::V_EMPTY + s), ((t / S) - 1) & 1, abort_flag, p.status,
                                 site + C::V_EMPTY + s)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::V_FULL + s), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(sV + s * C::KV_BYTES + c * C::KV_CHUNK, &p.tm_v, bar(C::V_FULL + s), 64 * c,
                        w.h, j * kWKeys, w.b);
        }
        __syncwarp();
        ++v_issued;
      }
    }
    // every copy started must land before the CTA exits (waits that ignore the
    // abort flag; on the normal path they are complete)
    volatile int never = 0;
    if (q_cnt > 0) mbar_wait(bar(C::Q_FULL), (q_cnt - 1) & 1, &never, p.status, site + C::Q_FULL);
    for (int i = (k_issued > S ? k_issued - S : 0); i < k_issued; ++i) {
      mbar_wait(bar(C::K_FULL + i % S), (i / S) & 1, &never, p.status, site + C::K_FULL);
      if (i < v_issued)
        mbar_wait(bar(C::V_FULL + i % S), (i / S) & 1, &never, p.status, site + C::V_FULL);
    }
  } else if (warp == kWMmaWarp) {
    // ---- MMA issuer
    const int site = kRoleWMma * 64;
    const int n_ks = p.dk_steps;  // K16 steps of S = Q K^T (<= 16)
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kWKeys, false, false);
    const uint32_t idesc_o = idesc_bf16_f32(128, p.dv_n, false, true);
    // K tile: K-major (keys are rows of 128 B per 64-feature chunk, 8-row
    // groups 1024 B apart, +32 B per K16 step inside a chunk); V tile:
    // N-major (features contiguous, 64-feature chunks KV_CHUNK apart, +2048 B
    // per 16 keys)
    const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sV, C::KV_CHUNK, 1024);
    int u_cnt = 0, t = 0;
    bool ok = true;
    auto issue_s = [&](int tt, bool last) {
      const int s = tt % S;
      if (!mbar_wait(bar(C::K_FULL + s), (tt / S) & 1, abort_flag, p.status, site + C::K_FULL + s))
        return false;
      tc_fence_after();
      const uint32_t d = tmem + ((tt & 1) ? C::TM_S1 : C::TM_S0);
      const uint64_t b = dk0 + static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          if (ks >= n_ks) break;
          const uint64_t off =
              static_cast<uint64_t>((((ks >> 2) * C::KV_CHUNK) + (ks & 3) * 32) >> 4);
          umma_ts(d, tmem + C::TM_Q + 8u * ks, b + off, idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(bar(C::S_FULL + (tt & 1)));
        umma_commit(bar(C::K_EMPTY + s));
        if (last) umma_commit(bar(C::Q_TMEM_FREE));
      }
      __syncwarp();
      return true;
    };
    auto issue_pv = [&](int tt, bool first, bool last) {
      const int s = tt % S;
      if (!mbar_wait(bar(C::P_FULL + (tt & 1)), (tt >> 1) & 1, abort_flag, p.status,
                     site + C::P_FULL + (tt & 1)) ||
          !mbar_wait(bar(C::V_FULL + s), (tt / S) & 1, abort_flag, p.status, site + C::V_FULL + s))
        return false;
      // the previous unit's epilogue must have read O before it is overwritten
      if (first && u_cnt > 0 &&
          !mbar_wait(bar(C::O_FREE), (u_cnt - 1) & 1, abort_flag, p.status, site + C::O_FREE))
        return false;
      tc_fence_after();
      const uint32_t a = tmem + ((tt & 1) ? C::TM_S1 : C::TM_S0);
      const uint64_t b = dv0 + static_cast<uint64_t>((s * C::KV_BYTES) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < kWKeys / 16; ++ks)
          umma_ts(tmem + C::TM_O, a + 8u * ks, b + static_cast<uint64_t>((ks * 2048) >> 4),
                  idesc_o, (ks > 0 || !first) ? 1u : 0u);
        umma_commit(bar(C::PV_DONE));
        umma_commit(bar(C::V_EMPTY + s));
        if (last) umma_commit(bar(C::O_DONE));
      }
      __syncwarp();
      return true;
    };
    for (int k = 0; ok; ++k) {
      const int u = next_unit(k, kRoleWMma);
      if (u < 0) break;
      const WUnit w = wide_unit(p, u);
      if (w.n == 0) continue;
      if (!mbar_wait(bar(C::Q_TMEM_FULL), u_cnt & 1, abort_flag, p.status, site + C::Q_TMEM_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S(0), then per tile S(j+1) before PV(j)
      ok = issue_s(t, w.n == 1);
      for (int j = 0; ok && j < w.n; ++j) {
        if (j + 1 < w.n) ok = issue_s(t + j + 1, j + 2 == w.n);
        if (ok) ok = issue_pv(t + j, j == 0, j + 1 == w.n);
      }
      t += w.n;
      ++u_cnt;
    }
    // every MMA issued completes before TMEM is released
    if (elect_one()) umma_commit(bar(C::DRAIN));
    __syncwarp();
    volatile int never = 0;
    mbar_wait(bar(C::DRAIN), 0, &never, p.status, site + C::DRAIN);
  } else if (warp < 4) {
    // ---- softmax + epilogue (thread = query row)
    const int site = kRoleWSoftmax * 64;
    const int row = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c2 = p.scale_log2;
    const int dv_n = p.dv_n;
    const uint32_t out_base = sOut + static_cast<uint32_t>(warp * 2 * C::OUT_CHUNK);
    int q_copies = 0, o_cnt = 0, t = 0, chunks = 0;
    bool prev_stored = true;  // the previous chunk issued a TMA store
    bool ok = true;
    // Copies this thread's row of a unit's Q (256 bf16, 128-byte swizzle)
    // from the staging buffer into TMEM, once the last S of the previous unit
    // with key tiles no longer reads TMEM's Q.
    auto copy_q = [&]() -> bool {
      if (!mbar_wait(bar(C::Q_FULL), q_copies & 1, abort_flag, p.status, site + C::Q_FULL) ||
          (q_copies > 0 && !mbar_wait(bar(C::Q_TMEM_FREE), (q_copies - 1) & 1, abort_flag,
                                      p.status, site + C::Q_TMEM_FREE)))
        return false;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = ld_shared_v4(sQ + c * C::Q_CHUNK + row * 128 +
                                       (static_cast<uint32_t>(v ^ (row & 7)) << 4));
          r[4 * v] = x.x;
          r[4 * v + 1] = x.y;
          r[4 * v + 2] = x.z;
          r[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + C::TM_Q + 32u * c, r);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::Q_TMEM_FULL));
      mbar_arrive(bar(C::Q_STAGE_FREE));
      ++q_copies;
      return true;
    };
    int u = next_unit(0, kRoleWSoftmax);
    WUnit w{};
    if (u >= 0) {
      w = wide_unit(p, u);
      if (w.n > 0) ok = copy_q();
    }
    for (int k = 0; ok && u >= 0; ++k) {
      const int qi = w.q0 + row;
      float m_ref = 0.f, l = 0.f;
      for (int j = 0; j < w.n; ++j, ++t) {
        const int buf = t & 1;
        if (!mbar_wait(bar(C::S_FULL + buf), (t >> 1) & 1, abort_flag, p.status,
                       site + C::S_FULL + buf)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + (buf ? C::TM_S1 : C::TM_S0);
        float x[64];
        {
          uint32_t r[64];
          tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld32(tS + 32u, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(r[c]);
        }
        const int kbase = j * kWKeys;
        int lim = w.kv_len - kbase;
        if (masks_causal(p.mask_kind) && qi - kbase + 1 < lim) lim = qi - kbase + 1;
        if (lim < kWKeys) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
        float mk[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mk[q] = fmaxf(x[2 * q], x[2 * q + 1]);
#pragma unroll
        for (int c = 16; c < 64; c += 16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) mk[q] = fmax3(mk[q], x[c + 2 * q], x[c + 2 * q + 1]);
        }
        const float mx =
            fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7])) * c2;
        bool move = false;
        float alpha = 1.f;
        if (j == 0) {
          m_ref = (mx == -INFINITY) ? 0.f : mx;
        } else if (mx > m_ref + kWRescaleThreshold) {
          move = true;
          alpha = ex2_approx(m_ref - mx);
          l *= alpha;
          m_ref = mx;
        }
        const float nm = -m_ref;
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          fma2(x[c], x[c + 1], x[c], x[c + 1], c2, c2, nm, nm);
          x[c] = ex2_approx(x[c]);
          x[c + 1] = ex2_approx(x[c + 1]);
          const int q = (c >> 1) & 3;
          add2(sa[q], sb[q], sa[q], sb[q], x[c], x[c + 1]);
          pk[c >> 1] = pack_bf16x2(x[c], x[c + 1]);
        }
        add2(sa[0], sb[0], sa[0], sb[0], sa[1], sb[1]);
        add2(sa[2], sb[2], sa[2], sb[2], sa[3], sb[3]);
        l += (sa[0] + sb[0]) + (sa[2] + sb[2]);
        if (__any_sync(0xffffffffu, move)) {
          // O holds PV(t - 1) only once that product is complete
          if (t > 0 && !mbar_wait(bar(C::PV_DONE), (t - 1) & 1, abort_flag, p.status,
                                  site + C::PV_DONE)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c32 = 0; c32 < W / 32; ++c32) {
            if (32 * c32 >= dv_n) break;
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + C::TM_O + 32u * c32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float a0, a1;
              mul2(a0, a1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha);
              o[i] = __float_as_uint(a0);
              o[i + 1] = __float_as_uint(a1);
            }
            tmem_st32(tmem + lane_off + C::TM_O + 32u * c32, o);
          }
        }
        tmem_st32(tS, pk);
        tmem_st_wait();
        tc_fence_before();
        // (test hook: the CTA's first weights are never handed over, so the
        // MMA warp's bounded wait runs out)
        if (!(p.withhold_p && k == 0 && j == 0)) mbar_arrive(bar(C::P_FULL + buf));
      }
      if (!ok) break;
      // The next unit's Q goes into TMEM now (this unit's last S is complete:
      // its scores were read), so the MMA warp computes the next unit's first
      // scores while this unit's epilogue runs.
      const int u_next = next_unit(k + 1, kRoleWSoftmax);
      WUnit w_next{};
      if (u_next >= 0) {
        w_next = wide_unit(p, u_next);
        if (w_next.n > 0 && !copy_q()) {
          ok = false;
          break;
        }
      }
      // ---- epilogue: O / l to bf16, this warp's 32 rows, 64 columns at a time
      // through the warp's staging buffers and a TMA store
      if (w.n > 0) {
        if (!mbar_wait(bar(C::O_DONE), o_cnt & 1, abort_flag, p.status, site + C::O_DONE)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      if (p.lse && qi < p.Lq)
        p.lse[(static_cast<size_t>(w.b) * p.H + w.h) * p.Lq + qi] =
            (l > 0.f) ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      const int n_chunks = (dv_n + 63) / 64;
      for (int c = 0; c < n_chunks; ++c, ++chunks) {
        const uint32_t stage = out_base + static_cast<uint32_t>((chunks & 1) * C::OUT_CHUNK);
        // the store issued from this buffer two chunks ago must have read it
        // (at most one group still reading when the previous chunk stored,
        // none when it stored nothing)
        if (lane == 0) {
          if (prev_stored) {
            tma_store_wait_read_1();
          } else {
            tma_store_wait_read();
          }
        }
        __syncwarp();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t o[32];
          const bool written = 64 * c + 32 * half < dv_n;
          if (w.n > 0 && written) {
            tmem_ld32(tmem + lane_off + C::TM_O + 64u * c + 32u * half, o);
            tmem_ld_wait();
            if (c == n_chunks - 1 && (half == 1 || 64 * c + 32 >= dv_n)) {
              tc_fence_before();
              mbar_arrive(bar(C::O_FREE));  // O may take the next unit's products
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint32_t wd[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              wd[i] = pack_bf16x2(__uint_as_float(o[8 * v4 + 2 * i]) * inv,
                                  __uint_as_float(o[8 * v4 + 2 * i + 1]) * inv);
            const uint32_t unit16 = static_cast<uint32_t>(4 * half + v4);
            st_shared_v4(stage + lane * 128 + ((unit16 ^ (lane & 7)) << 4), wd[0], wd[1], wd[2],
                         wd[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        // (a warp whose 32 rows all lie past Lq stores nothing)
        prev_stored = w.q0 + 32 * warp < p.Lq;
        if (lane == 0 && prev_stored) {
          tma_store_4d(&p.tm_o, stage, 64 * c, w.h, w.q0 + 32 * warp, w.b);
          tma_store_commit();
        }
        __syncwarp();
      }
      if (w.n > 0) ++o_cnt;
      u = u_next;
      w = w_next;
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  } else if (warp == kWSchedulerWarp && lane == 0) {
    // ---- scheduler: publishes this CTA's own unit, then keeps one unit of
    // look-ahead by cancelling CTAs that have not started and taking theirs
    int unit = static_cast<int>(blockIdx.x);
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      if (k >= 2 && !mbar_wait(bar(C::UNIT_EMPTY + slot), ((k >> 1) - 1) & 1, abort_flag,
                               p.status, kRoleWScheduler * 64 + C::UNIT_EMPTY + slot))
        unit = -1;
      unit_slot[slot] = unit;
      mbar_arrive(bar(C::UNIT_FULL + slot));
      if (unit < 0) break;
      mbar_arrive_expect_tx(bar(C::CLC), 16);
      clc_try_cancel(clc_resp, bar(C::CLC));
      // the response lands asynchronously: wait for it even when giving up,
      // so nothing is written to shared memory after the CTA exits
      volatile int never = 0;
      if (!mbar_wait(bar(C::CLC), k & 1, &never, p.status, kRoleWScheduler * 64 + C::CLC) ||
          *abort_flag) {
        unit = -1;
      } else {
        unit = clc_query_first_ctaid_x(clc_resp);  // -1 when nothing was cancelled
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int W>
cudaError_t launch_wide_w(const Bf16Params& params, cudaStream_t stream, LaunchInfo* info) {
  using C = WCfg<W>;
  Bf16Params p = params;
  {
    // heads whose K/V stay in L2 while their query tiles run
    const long long per_head = 2ll * p.Lk * W * 2 > 0 ? 2ll * p.Lk * W * 2 : 1;
    long long hg = kWHeadGroupBytes / per_head;
    const long long bh = static_cast<long long>(p.B) * p.H;
    if (hg > bh) hg = bh;
    if (hg < 1) hg = 1;
    p.head_group = static_cast<int>(hg);
  }
  p.n_qtiles = (p.Lq + kBlockM - 1) / kBlockM;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(fwd_wide_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long units = static_cast<long long>(p.B) * p.H * p.n_qtiles;
  if (units <= 0 || units > 0x7fffffffll) return cudaErrorInvalidValue;
  // one CTA per unit; running CTAs take over the units of those not started
  const int grid = static_cast<int>(units);
  e = launch_serialized(fwd_wide_kernel<W>, dim3(grid), dim3(kWThreads), C::SMEM, stream, p);
  if (e != cudaSuccess) return e;
  if (info) {
    info->kernels = 1;
    info->grid = grid;
    info->block = kWThreads;
    info->smem = C::SMEM;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_wide(const Bf16Params& params, int width, cudaStream_t stream,
                            LaunchInfo* info) {
  if (width == 256) return launch_wide_w<256>(params, stream, info);
  if (width == 64) return launch_wide_w<64>(params, stream, info);
  return cudaErrorInvalidValue;
}

}  // namespace mha
