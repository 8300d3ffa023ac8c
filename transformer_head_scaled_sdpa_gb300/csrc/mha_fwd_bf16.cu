// mha_fwd_bf16.cu -- bf16 attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Computes, for every (sequence b, head h) and every 256-query block, the
// rows of
//   O = softmax(Q K^T * scale) V
// ("Attention Is All You Need", Section 3.2.1, Equation (1); all heads in
// parallel, Section 3.2.2) without writing the score matrix to memory: K/V
// are streamed in 128-key tiles and the softmax is evaluated online.  Each
// query row keeps a reference maximum m and a running sum l; a tile's
// probabilities are p = 2^(s * scale * log2(e) - m), and the partial output
// and l are rescaled by 2^(m_old - m_new) when m moves.  Any reference value
// gives the same weights, because adding one constant to all scores of a row
// leaves the weights unchanged (formula page transformer-attention, section
// 証明, weight-ratio step); m only has to keep p within range.  So a row's m
// is moved only when a tile's maximum exceeds it by more than 8 (log2 units:
// p <= 2^8, well inside bf16's range, float32 sums), which makes rescaling
// rare.
//
// Work unit: (b, h, two 128-row query tiles Q0, Q1) sharing every K/V tile.
// The grid has one CTA per unit, but CTAs are persistent: once a running CTA
// has its own unit it cancels a CTA that has not started yet (cluster launch
// control) and processes that CTA's unit too, so each SM keeps one CTA whose
// set-up, tensor memory and pipelines carry over from unit to unit, the next
// unit's Q is loaded while the current one finishes, and the hardware's
// launch order (heavy causal blocks first) still balances the load.
// Paired units (d_k = 64, at most 128 query rows, more heads than SMs): a
// unit is instead one 128-row query tile of two heads, Q0 of one and Q1 of
// the next, each with its own K/V tiles in the ring, so no softmax warpgroup
// idles for want of a second query tile and the grid halves.
//
// 384 threads (three warpgroups) in five roles:
//   warps 0-3   softmax + epilogue for Q0 (thread r owns row r = TMEM lane r)
//   warps 4-7   softmax + epilogue for Q1
//   warp 8      TMEM allocator and MMA issuer (for Q0 only with d_k = 64)
//   warp 11     MMA issuer for Q1 (d_k = 64; idle with d_k = 128)
//   warp 9      TMA producer: Q0, Q1, then K_j / V_j into an NS-stage ring
//   warp 10     scheduler: feeds a two-slot queue of decoded units to the others
// The third warpgroup gives registers to the softmax warpgroups, which hold
// a whole 128-score row per thread: launched at 168 per thread, it drops to
// 112 and they rise to 192 (256*192 + 128*112 = 63488 <= 384*168 registers).
// TMEM (512 columns), d_k = 128: S0 | S1 | O0 | O1.  Softmax g reads S_g
// (float32), writes P_g as bf16 pairs into the first 64 columns of S_g, and
// the P.V MMA reads P_g from TMEM.  Per key tile j the MMA warp issues
//   PV0(j), S0(j+1), PV1(j), S1(j+1)
// so softmax 0 works on S0(j+1) while the tensor core runs PV1(j) and
// S1(j+1), and vice versa.  MMAs of one thread run in issue order, so
// S_g(j+1) overwrites P_g(j) only after PV_g(j) has read it, and once S_g(j+1)
// is complete PV_g(j) is too: softmax g may rescale O_g in place then.
// d_k = 64: S0 | S1 | O0 | O1 | P0 | P1.  Softmax g releases S_g as soon as it
// has read it, so MMA warp g issues S_g(j+1) before PV_g(j) and the next
// scores are ready when softmax g finishes a tile; softmax g waits for
// PV_g(j-1) only before it rewrites P_g (and rescales O_g).
// Masks: causal tiles above the diagonal are never loaded or computed; the
// diagonal tile and a ragged last key tile are masked per element (score set
// to -inf, weight exactly 0: formula page, 応用, 先を読まない仕掛け).
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

constexpr int kThreads = 384;
// warp roles: softmax warps 0-3 (Q0) and 4-7 (Q1), then the third warpgroup
constexpr int kSoftmaxWarp0 = 0;
constexpr int kMmaWarp = 8, kProducerWarp = 9, kMma1Warp = 11;  // warp 10: scheduler
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p stays <= 2^8
// Heads dispatched together are chosen by their K/V bytes, about this much
// per group, so a group's K/V stay in L2 while its query blocks run (48 heads
// of the GPT-3-like shape, 96 of big16 L 2048, every head of the base-model
// shapes).  Measured against 32 MiB: GPT-3-like +2 % in short runs and +1.5 %
// in 2000-call runs under the power cap, the d_k 64 workloads -0.3 % to +1 %;
// 64 MiB fell in between; 128 MiB was faster still in short runs but doubled
// the GPT-3-like kernel's DRAM reads and lost 5 % under the power cap.
constexpr long long kHeadGroupBytes = 48ll << 20;
// unit-queue readers: 8 softmax warps, the producer and 1 or 2 MMA warps
template <int D>
constexpr int unit_consumers() { return D == 64 ? 11 : 10; }

template <int D>
struct Cfg {
  static constexpr int KCH = D / 64;             // 128-byte chunks along d
  static constexpr int CHUNK = 128 * 128;        // one [128 rows x 128 B] swizzled chunk
  static constexpr int TILE = KCH * CHUNK;       // one 128-row Q, K or V tile
  static constexpr int NS = (D == 64) ? 4 : 2;   // K/V ring stages
  static constexpr int OFF_Q = 0;                // Q0, Q1
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_STAGE = OFF_V + NS * TILE;  // epilogue staging, one CHUNK per softmax warpgroup
  static constexpr int OFF_BAR = OFF_STAGE + 2 * CHUNK;
  static constexpr int NBAR = 31 + 4 * NS;
  // tmem slot (+0), abort flag (+4), unit queue (+8, +12), CLC response (+16,
  // 16 bytes, must be 16-byte aligned), then the queue's two decoded units
  // (64 bytes each)
  static constexpr int OFF_MISC = (OFF_BAR + 8 * NBAR + 63) / 64 * 64;
  static constexpr int OFF_CLC = OFF_MISC + 16;
  static constexpr int OFF_UNITS = OFF_MISC + 64;
  static constexpr int SMEM = OFF_UNITS + 128 + 1024;  // + slack to align the base to 1024
  // TMEM columns.  With d_k = 64 P has columns of its own (S0 | S1 | O0 | O1 |
  // P0 | P1), so S_g(j+1) can be computed while softmax g still works on tile
  // j; with d_k = 128 the 512 columns hold only S0 | S1 | O0 | O1 and P_g is
  // written over the first 64 columns of S_g.
  static constexpr bool SEPARATE_P = (D == 64);
  // With two stages (d_k = 128) a stage's K tile is released after its last S
  // MMA and its V tile after its last P.V MMA, which gives each load about
  // one key tile of lead time; with four (d_k = 64) one release per stage
  // (K_EMPTY) covers both.
  static constexpr bool SPLIT_RELEASE = (NS == 2);
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128;
  static constexpr uint32_t TM_O0 = 256, TM_O1 = 256 + D;
  static constexpr uint32_t TM_P0 = SEPARATE_P ? 384 : TM_S0, TM_P1 = SEPARATE_P ? 448 : TM_S1;
  static constexpr uint32_t TMEM_COLS = 512;
  // registers per thread after rebalancing (softmax warpgroups, the rest)
  static constexpr uint32_t REGS_SOFTMAX = 192;
  static constexpr uint32_t REGS_OTHER = 112;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(OFF_BAR % 8 == 0 && OFF_CLC % 16 == 0, "barrier / response alignment");
  static_assert(OFF_Q % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0 &&
                    OFF_STAGE % 1024 == 0,
                "128-byte-swizzled tiles need 1024-byte alignment");
  static_assert(256 * REGS_SOFTMAX + 128 * REGS_OTHER <= kThreads * 168, "register split");
};

// barrier ids inside the barrier block
template <int NS>
struct Bars {
  static constexpr int Q_FULL = 0;                // + g: Q_g landed
  static constexpr int Q_FREE = 2;                // + g: last S_g of the unit done (Q_g reusable)
  static constexpr int S_FULL = 4;                // + g: S_g in TMEM
  static constexpr int P_FULL = 6;                // + g: P_g in TMEM (128 arrivals)
  static constexpr int O_DONE = 8;                // + g: last PV_g of the unit done
  static constexpr int O_FREE = 10;               // + g: epilogue read O_g (128 arrivals)
  static constexpr int UNIT_FULL = 12;            // + slot: unit published
  static constexpr int UNIT_EMPTY = 14;           // + slot: all consumers read it
  static constexpr int CLC = 16;                  // cancellation response landed
  static constexpr int S_FREE = 17;               // + g: softmax read S_g (128 arrivals; separate P only)
  static constexpr int PV_DONE = 19;              // + g: PV_g done (separate P only)
  static constexpr int DRAIN = 21;                // + g: MMA warp g's operations complete
  static constexpr int K_FULL = 23;               // + stage
  static constexpr int V_FULL = 23 + NS;          // + stage
  static constexpr int K_EMPTY = 23 + 2 * NS;     // + stage: its K tile's last S MMA done (or,
                                                  // without split release, the whole stage:
                                                  // 2 arrivals, one per MMA warp)
  static constexpr int V_EMPTY = 23 + 3 * NS;     // + stage: its V tile's last P.V MMA done
  static constexpr int TOK_A = 23 + 4 * NS;       // + quarter: Q0's warp may take its exponentials (32 arrivals)
  static constexpr int TOK_B = 27 + 4 * NS;       // + quarter: Q1's warp may take its exponentials (32 arrivals)
};

// role ids for the status "site" field
constexpr int kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleScheduler = 4;

// A shared unit: (b, h, 256-row block), two query tiles of one head sharing
// every K/V tile; ring slot j holds key tile j for both.
struct SharedUnit {
  int b, h;
  int q0;       // first query row of Q0
  int n[2];     // key tiles for Q0, Q1
  int kv_len;   // keys visible before the causal limit
  __device__ __forceinline__ int seq(int) const { return b; }
  __device__ __forceinline__ int head(int) const { return h; }
  __device__ __forceinline__ int qstart(int g) const { return q0 + g * kBlockM; }
  __device__ __forceinline__ int keys(int) const { return kv_len; }
  __device__ __forceinline__ void store(volatile int* w) const {
    w[0] = b; w[1] = h; w[2] = q0; w[3] = n[0]; w[4] = n[1]; w[5] = kv_len;
  }
  __device__ __forceinline__ void load(const volatile int* w) {
    b = w[0]; h = w[1]; q0 = w[2]; n[0] = w[3]; n[1] = w[4]; kv_len = w[5];
  }
};

// A paired unit: (two consecutive heads, 128-row query tile), Q_g from head
// 2i + g with key tiles of its own.  The heads' tiles alternate in the ring
// (Q0's tile j, Q1's tile j, ...) while both have tiles, then the longer list
// goes on alone.  Per-tile fields are read by select, not by index: g is
// often not a compile-time constant, and an indexed struct would live in
// local memory.
struct PairedUnit {
  int b[2], h[2];
  int qs[2];        // first query row of Q_g (Lq: no such tile)
  int n[2];         // key tiles of Q_g
  int kv_len[2];
  int m;            // min(n[0], n[1])
  __device__ __forceinline__ int seq(int g) const { return g ? b[1] : b[0]; }
  __device__ __forceinline__ int head(int g) const { return g ? h[1] : h[0]; }
  __device__ __forceinline__ int qstart(int g) const { return g ? qs[1] : qs[0]; }
  __device__ __forceinline__ int keys(int g) const { return g ? kv_len[1] : kv_len[0]; }
  __device__ __forceinline__ void store(volatile int* w) const {
    w[0] = b[0]; w[1] = b[1]; w[2] = h[0]; w[3] = h[1]; w[4] = qs[0]; w[5] = qs[1];
    w[6] = n[0]; w[7] = n[1]; w[8] = kv_len[0]; w[9] = kv_len[1]; w[10] = m;
  }
  __device__ __forceinline__ void load(const volatile int* w) {
    b[0] = w[0]; b[1] = w[1]; h[0] = w[2]; h[1] = w[3]; qs[0] = w[4]; qs[1] = w[5];
    n[0] = w[6]; n[1] = w[7]; kv_len[0] = w[8]; kv_len[1] = w[9]; m = w[10];
  }
  __device__ __forceinline__ int slots() const { return n[0] + n[1]; }
  // ring slot (within the unit) of Q_g's key tile j
  __device__ __forceinline__ int slot_of(int g, int j) const {
    return j < m ? 2 * j + g : 2 * m + (j - m);
  }
  // query tile owning a slot (returned) and its key tile *j
  __device__ __forceinline__ int owner(int slot, int* j) const {
    if (slot < 2 * m) {
      *j = slot >> 1;
      return slot & 1;
    }
    *j = m + (slot - 2 * m);
    return n[0] > n[1] ? 0 : 1;
  }
};

template <bool PAIRED>
struct UnitSel {
  using T = SharedUnit;
};
template <>
struct UnitSel<true> {
  using T = PairedUnit;
};

__device__ __forceinline__ int visible_keys(const Bf16Params& p, int b) {
  if (!masks_padding(p.mask_kind)) return p.Lk;
  const int len = __ldg(p.key_lens + b);
  return len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
}

// key tiles of the 128-row query tile starting at qs
__device__ __forceinline__ int tiles_for(const Bf16Params& p, int qs, int kv_len) {
  int n = (qs < p.Lq) ? (kv_len + kBlockN - 1) / kBlockN : 0;
  if (masks_causal(p.mask_kind) && n > qs / kBlockN + 1) n = qs / kBlockN + 1;
  return n;
}

// Units are ordered in groups of p.head_group heads, so a group's K/V stay in
// L2 while all of its query blocks run; inside a group the causal blocks go
// heaviest first.
template <bool PAIRED>
__device__ __forceinline__ typename UnitSel<PAIRED>::T decode_unit(const Bf16Params& p,
                                                                   int unit) {
  const int bh_count = p.B * p.H;
  const int n_blocks = p.n_qtiles;
  typename UnitSel<PAIRED>::T u;
  if constexpr (!PAIRED) {
    const int hg = p.head_group;
    const int group = unit / (hg * n_blocks);
    const int within = unit - group * hg * n_blocks;
    const int heads_here = min(hg, bh_count - group * hg);
    const int pair_idx = within / heads_here;
    const int bh = group * hg + within % heads_here;
    const int t = masks_causal(p.mask_kind) ? (n_blocks - 1 - pair_idx) : pair_idx;
    u.b = bh / p.H;
    u.h = bh % p.H;
    u.q0 = t * kUnitRows;
    int kv_len = p.Lk;
    if (masks_padding(p.mask_kind)) {
      const int len = __ldg(p.key_lens + u.b);
      kv_len = len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
    }
    u.kv_len = kv_len;
    const int n_kv = (kv_len + kBlockN - 1) / kBlockN;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int qs = u.q0 + g * kBlockM;
      int n = (qs < p.Lq) ? n_kv : 0;
      if (masks_causal(p.mask_kind) && n > qs / kBlockN + 1) n = qs / kBlockN + 1;
      u.n[g] = n;
    }
  } else {
    const int kPairGroup = p.head_group / 2;
    const int n_pairs = (bh_count + 1) / 2;
    const int group = unit / (kPairGroup * n_blocks);
    const int within = unit - group * kPairGroup * n_blocks;
    const int pairs_here = min(kPairGroup, n_pairs - group * kPairGroup);
    const int tile_idx = within / pairs_here;
    const int pair = group * kPairGroup + within % pairs_here;
    const int t = masks_causal(p.mask_kind) ? (n_blocks - 1 - tile_idx) : tile_idx;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      int bh = 2 * pair + g;
      const bool exists = bh < bh_count;  // an odd head count leaves the last Q1 empty
      if (!exists) bh = 2 * pair;
      u.b[g] = bh / p.H;
      u.h[g] = bh % p.H;
      u.qs[g] = exists ? t * kBlockM : p.Lq;
      u.kv_len[g] = visible_keys(p, u.b[g]);
      u.n[g] = tiles_for(p, u.qs[g], u.kv_len[g]);
    }
    u.m = min(u.n[0], u.n[1]);
  }
  return u;
}

// Per-CTA context shared by the roles.
struct Ctx {
  uint32_t sQ, sK, sV, sStage, s_bar;
  uint32_t tmem;
  uint32_t clc_resp;           // 16-byte cancellation response
  volatile int* abort_flag;
  volatile int* unit_slot;     // [2]
  volatile int* unit_data;     // [2][16]: the queued units, decoded
  int warp, lane;
  __device__ __forceinline__ uint32_t bar(int id) const {
    return s_bar + 8u * static_cast<uint32_t>(id);
  }
};

// Waits for the k-th unit of this CTA from the queue; returns its index, or
// -1 at the end of the work (or when the CTA gave up), and copies the unit,
// decoded by the scheduler, into u.  Every consumer calls it once per unit,
// in the same order.
template <int NS, typename UnitT>
__device__ __forceinline__ int next_unit(const Bf16Params& p, const Ctx& cx, int k, int role,
                                         bool arrive, UnitT& u) {
  using BA = Bars<NS>;
  const int slot = k & 1;
  if (!mbar_wait(cx.bar(BA::UNIT_FULL + slot), (k >> 1) & 1, cx.abort_flag, p.status,
                 role * 64 + BA::UNIT_FULL + slot))
    return -1;
  const int unit = cx.unit_slot[slot];
  if (unit >= 0) u.load(cx.unit_data + 16 * slot);
  __syncwarp();
  if (arrive) mbar_arrive(cx.bar(BA::UNIT_EMPTY + slot));
  return unit;
}

// For a consumer that decodes the unit itself.
struct UnitIndexOnly {
  __device__ __forceinline__ void load(const volatile int*) {}
};

// Scheduler (warp 10, one lane): publishes the CTA's own unit, then keeps one
// unit of look-ahead by cancelling not-yet-launched CTAs and taking their
// units, until no CTA is left to cancel.  It also decodes each unit for the
// other roles, off their critical paths (measured: the decode, with its
// integer divisions, took the MMA warp about 1200 cycles at each unit
// boundary, being issued between busy softmax warps).
template <int D, bool PAIRED>
__device__ __forceinline__ void scheduler_role(const Bf16Params& p, const Ctx& cx) {
  using BA = Bars<Cfg<D>::NS>;
  if (cx.lane != 0) return;
  int unit = static_cast<int>(blockIdx.x);
  for (int k = 0;; ++k) {
    const int slot = k & 1;
    if (k >= 2 && !mbar_wait(cx.bar(BA::UNIT_EMPTY + slot), ((k >> 1) - 1) & 1, cx.abort_flag,
                             p.status, kRoleScheduler * 64 + BA::UNIT_EMPTY + slot))
      unit = -1;
    if (unit >= 0) decode_unit<PAIRED>(p, unit).store(cx.unit_data + 16 * slot);
    cx.unit_slot[slot] = unit;
    mbar_arrive(cx.bar(BA::UNIT_FULL + slot));
    if (unit < 0) break;
    // ask for the next unit while this one runs
    mbar_arrive_expect_tx(cx.bar(BA::CLC), 16);
    clc_try_cancel(cx.clc_resp, cx.bar(BA::CLC));
    // the response is written asynchronously: wait for it even when the CTA
    // is giving up, so nothing lands in shared memory after exit
    volatile int never = 0;
    if (!mbar_wait(cx.bar(BA::CLC), k & 1, &never, p.status, kRoleScheduler * 64 + BA::CLC) ||
        *cx.abort_flag) {
      unit = -1;
    } else {
      unit = clc_query_first_ctaid_x(cx.clc_resp);  // -1 when nothing was cancelled
    }
  }
}

// TMA producer (warp 9): per unit Q0, K_0, Q1, V_0, then K_j / V_j into the
// ring.  The whole warp runs the loop and waits; one elected lane issues.
template <int D>
__device__ __forceinline__ void producer_role(const Bf16Params& p, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;
  int q_cnt[2] = {0, 0};  // Q_g loads so far
  int kv_cnt = 0;         // K/V tiles of the units before the current one
  int kv_issued = 0;      // K tile loads issued
  int v_issued = 0;       // V tile loads issued
  bool ok = true;
  for (int k = 0; ok; ++k) {
    typename UnitSel<false>::T u;
    const int unit = next_unit<NS>(p, cx, k, kRoleProducer, cx.lane == 0, u);
    if (unit < 0) break;
    const int n_max = max(u.n[0], u.n[1]);
    auto load_q = [&](int g) {
      // the previous unit's last S_g must be done with the Q_g buffer
      if (q_cnt[g] > 0 && !mbar_wait(cx.bar(BA::Q_FREE + g), (q_cnt[g] - 1) & 1, cx.abort_flag,
                                     p.status, kRoleProducer * 64 + BA::Q_FREE + g))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(cx.bar(BA::Q_FULL + g), C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(cx.sQ + g * C::TILE + c * C::CHUNK, &p.tm_q, cx.bar(BA::Q_FULL + g), 64 * c,
                      u.h, u.q0 + g * kBlockM, u.b);
      }
      __syncwarp();
      ++q_cnt[g];
      return true;
    };
    auto load_kv = [&](int j, bool is_v) {
      const int t = kv_cnt + j;
      const int s = t % NS;
      const uint32_t dst = (is_v ? cx.sV : cx.sK) + s * C::TILE;
      const uint32_t full = cx.bar((is_v ? BA::V_FULL : BA::K_FULL) + s);
      // the stage's previous K (or V) tile must be done with
      const int empty = (is_v ? BA::V_EMPTY : BA::K_EMPTY) + s;
      if (t >= NS && (!is_v || C::SPLIT_RELEASE) &&
          !mbar_wait(cx.bar(empty), ((t / NS) - 1) & 1, cx.abort_flag, p.status,
                     kRoleProducer * 64 + empty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(full, C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(dst + c * C::CHUNK, is_v ? &p.tm_v : &p.tm_k, full, 64 * c, u.h,
                      j * kBlockN, u.b);
      }
      __syncwarp();
      if (is_v) {
        ++v_issued;
      } else {
        ++kv_issued;
      }
      return true;
    };
    if (n_max == 0) continue;
    ok = (u.n[0] == 0 || load_q(0)) && load_kv(0, false) && (u.n[1] == 0 || load_q(1)) &&
         load_kv(0, true);
    for (int j = 1; ok && j < n_max; ++j) ok = load_kv(j, false) && load_kv(j, true);
    kv_cnt += n_max;
  }
  // Leave only when every copy this warp started has landed (the normal path
  // finds them complete already): the last Q_g and the last load of each
  // stage.  These waits ignore the abort flag: a copy still in flight must not
  // land in the shared memory of a CTA that has exited.
  volatile int never = 0;
  for (int g = 0; g < 2; ++g)
    if (q_cnt[g] > 0)
      mbar_wait(cx.bar(BA::Q_FULL + g), (q_cnt[g] - 1) & 1, &never, p.status,
                kRoleProducer * 64 + BA::Q_FULL + g);
  for (int t = (kv_issued > NS ? kv_issued - NS : 0); t < kv_issued; ++t) {
    const int s = t % NS;
    mbar_wait(cx.bar(BA::K_FULL + s), (t / NS) & 1, &never, p.status,
              kRoleProducer * 64 + BA::K_FULL + s);
    if (t < v_issued)
      mbar_wait(cx.bar(BA::V_FULL + s), (t / NS) & 1, &never, p.status,
                kRoleProducer * 64 + BA::V_FULL + s);
  }
}

// TMA producer for paired units: Q0 with its first K and V, Q1 with its
// first K and V, then the unit's ring slots in order.
template <int D>
__device__ __forceinline__ void producer_role_paired(const Bf16Params& p, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;
  int q_cnt[2] = {0, 0};  // Q_g loads so far
  int kv_cnt = 0;         // ring slots of the units before the current one
  int kv_issued = 0;      // K tile loads issued
  int v_issued = 0;       // V tile loads issued
  bool ok = true;
  for (int k = 0; ok; ++k) {
    typename UnitSel<true>::T u;
    const int unit = next_unit<NS>(p, cx, k, kRoleProducer, cx.lane == 0, u);
    if (unit < 0) break;
    auto load_q = [&](int g) {
      // the previous unit's last S_g must be done with the Q_g buffer
      if (q_cnt[g] > 0 && !mbar_wait(cx.bar(BA::Q_FREE + g), (q_cnt[g] - 1) & 1, cx.abort_flag,
                                     p.status, kRoleProducer * 64 + BA::Q_FREE + g))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(cx.bar(BA::Q_FULL + g), C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(cx.sQ + g * C::TILE + c * C::CHUNK, &p.tm_q, cx.bar(BA::Q_FULL + g), 64 * c,
                      u.head(g), u.qstart(g), u.seq(g));
      }
      __syncwarp();
      ++q_cnt[g];
      return true;
    };
    // key tile j of query tile g's head into ring slot `slot` of the unit
    auto load_kv = [&](int slot, int g, int j, bool is_v) {
      const int t = kv_cnt + slot;
      const int s = t % NS;
      const uint32_t dst = (is_v ? cx.sV : cx.sK) + s * C::TILE;
      const uint32_t full = cx.bar((is_v ? BA::V_FULL : BA::K_FULL) + s);
      // the stage's previous K (or V) tile must be done with
      const int empty = (is_v ? BA::V_EMPTY : BA::K_EMPTY) + s;
      if (t >= NS && (!is_v || C::SPLIT_RELEASE) &&
          !mbar_wait(cx.bar(empty), ((t / NS) - 1) & 1, cx.abort_flag, p.status,
                     kRoleProducer * 64 + empty))
        return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(full, C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(dst + c * C::CHUNK, is_v ? &p.tm_v : &p.tm_k, full, 64 * c, u.head(g),
                      j * kBlockN, u.seq(g));
      }
      __syncwarp();
      if (is_v) {
        ++v_issued;
      } else {
        ++kv_issued;
      }
      return true;
    };
    const int n_slots = u.slots();
    for (int slot = 0; ok && slot < n_slots; ++slot) {
      int j = 0;
      const int g = u.owner(slot, &j);
      ok = (j > 0 || load_q(g)) && load_kv(slot, g, j, false) && load_kv(slot, g, j, true);
    }
    kv_cnt += n_slots;
  }
  // Leave only when every copy this warp started has landed (the normal path
  // finds them complete already): the last Q_g and the last load of each
  // stage.  These waits ignore the abort flag: a copy still in flight must not
  // land in the shared memory of a CTA that has exited.
  volatile int never = 0;
  for (int g = 0; g < 2; ++g)
    if (q_cnt[g] > 0)
      mbar_wait(cx.bar(BA::Q_FULL + g), (q_cnt[g] - 1) & 1, &never, p.status,
                kRoleProducer * 64 + BA::Q_FULL + g);
  for (int t = (kv_issued > NS ? kv_issued - NS : 0); t < kv_issued; ++t) {
    const int s = t % NS;
    mbar_wait(cx.bar(BA::K_FULL + s), (t / NS) & 1, &never, p.status,
              kRoleProducer * 64 + BA::K_FULL + s);
    if (t < v_issued)
      mbar_wait(cx.bar(BA::V_FULL + s), (t / NS) & 1, &never, p.status,
                kRoleProducer * 64 + BA::V_FULL + s);
  }
}

// MMA issuer for one query tile, used with separate P (d_k = 64): warp 8
// serves Q0 and warp 11 Q1 (GSEL 0 and 1), each following only its own tile's
// chain so neither waits on the other's softmax; both release every K/V stage
// (the stage barrier counts two arrivals).  (With P over S, d_k = 128, one
// warp serves both tiles in a fixed ping-pong order: mma_role_pair.)  The
// whole warp runs the loop and the waits; one elected lane issues every
// tcgen05.mma and tcgen05.commit, with descriptors built once and stepped by
// constants.
template <int D, int GSEL, bool PAIRED, bool NARROW>
__device__ __forceinline__ void mma_role(const Bf16Params& p, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
  // NARROW: the head's own widths, ceil(d_k / 16) K steps for S and N = d_v
  // rounded up to 16 for P.V (features past d_k read as zero; O columns past
  // d_v unused); otherwise the kernel's full width, as compile-time constants
  const int n_ks = NARROW ? p.dk_steps : D / 16;
  const uint32_t idesc_o =
      NARROW ? idesc_bf16_f32(128, p.dv_n, false, true) : idesc_bf16_f32(128, D, false, true);
  // K-major Q and K tiles: 8-row groups 1024 B apart; V MN-major with its
  // second 64-wide d chunk one CHUNK further.
  const uint64_t dq0 = smem_desc_sw128(cx.sQ, 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(cx.sK, 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(cx.sV, C::CHUNK, 1024);
  const int site = kRoleMma * 64;
  auto commit = [&](int id) {
    if (elect_one()) umma_commit(cx.bar(id));
    __syncwarp();
  };
  // per query tile g: units with Q_g, P_g tiles consumed, S_g tiles issued,
  // units with O_g
  int q_cnt[2] = {0, 0}, s_cnt[2] = {0, 0}, s_iss[2] = {0, 0}, o_cnt[2] = {0, 0};
  int kv_cnt = 0;
  bool ok = true;
  // S_g = Q_g K_t^T (M 128 queries, N 128 keys, K = d in steps of 16) for the
  // unit's key tile j; with separate P the softmax must first have read the
  // previous S_g (any unit).  The last S_g of a unit frees Q_g.
  auto next_s = [&](int g, int t, int j, int n) {
    if constexpr (C::SEPARATE_P) {
      if (s_iss[g] > 0 && !mbar_wait(cx.bar(BA::S_FREE + g), (s_iss[g] - 1) & 1, cx.abort_flag,
                                     p.status, site + BA::S_FREE + g))
        return false;
    }
    if (!mbar_wait(cx.bar(BA::K_FULL + t % NS), (t / NS) & 1, cx.abort_flag, p.status,
                   site + BA::K_FULL + t % NS))
      return false;
    tc_fence_after();
    const uint64_t a = dq0 + static_cast<uint64_t>((g * C::TILE) >> 4);
    const uint64_t b = dk0 + static_cast<uint64_t>(((t % NS) * C::TILE) >> 4);
    const uint32_t tm_s = cx.tmem + (g ? C::TM_S1 : C::TM_S0);
    if (elect_one()) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        if (ks >= n_ks) break;
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ss(tm_s, a + off, b + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(cx.bar(BA::S_FULL + g));
      if (j + 1 == n) umma_commit(cx.bar(BA::Q_FREE + g));
    }
    __syncwarp();
    ++s_iss[g];
    return true;
  };
  // O_g += P_g V_t (A = P_g from TMEM, 16 keys = 8 columns per step; B = V_t
  // MN-major, 16 keys = 16 rows of 128 B per step); the unit's last PV_g
  // releases O_g to the epilogue.
  auto next_pv = [&](int g, int t, int j, int n) {
    const int s = t % NS;
    if (!mbar_wait(cx.bar(BA::P_FULL + g), s_cnt[g] & 1, cx.abort_flag, p.status,
                   site + BA::P_FULL + g) ||
        !mbar_wait(cx.bar(BA::V_FULL + s), (t / NS) & 1, cx.abort_flag, p.status,
                   site + BA::V_FULL + s))
      return false;
    // the previous unit's epilogue must have read O_g before it is overwritten
    if (j == 0 && o_cnt[g] > 0 &&
        !mbar_wait(cx.bar(BA::O_FREE + g), (o_cnt[g] - 1) & 1, cx.abort_flag, p.status,
                   site + BA::O_FREE + g))
      return false;
    ++s_cnt[g];
    tc_fence_after();
    const uint64_t b = dv0 + static_cast<uint64_t>((s * C::TILE) >> 4);
    const uint32_t tm_p = cx.tmem + (g ? C::TM_P1 : C::TM_P0);
    const uint32_t tm_o = cx.tmem + (g ? C::TM_O1 : C::TM_O0);
    if (elect_one()) {
#pragma unroll
      for (int ks = 0; ks < kBlockN / 16; ++ks)
        umma_ts(tm_o, tm_p + 8u * ks, b + static_cast<uint64_t>((ks * 2048) >> 4), idesc_o,
                (ks > 0 || j > 0) ? 1u : 0u);
      if constexpr (C::SEPARATE_P) umma_commit(cx.bar(BA::PV_DONE + g));
      if (j + 1 == n) umma_commit(cx.bar(BA::O_DONE + g));
    }
    __syncwarp();
    if (j + 1 == n) ++o_cnt[g];
    return true;
  };
  static_assert(GSEL == 0 || GSEL == 1, "one query tile per warp");
  static_assert(C::SEPARATE_P && !C::SPLIT_RELEASE,
                "one MMA warp per query tile: P apart from S, one release per stage");
  if constexpr (!PAIRED) {
    constexpr int g_lo = GSEL;
    constexpr int g_hi = GSEL;
    for (int k = 0; ok; ++k) {
      typename UnitSel<PAIRED>::T u;
      const int unit = next_unit<NS>(p, cx, k, kRoleMma, cx.lane == 0, u);
      if (unit < 0) break;
      const int n_max = max(u.n[0], u.n[1]);
      if (n_max == 0) continue;
      // prologue: S_g(0)
#pragma unroll
      for (int g = g_lo; g <= g_hi; ++g)
        if (ok && u.n[g] > 0)
          ok = mbar_wait(cx.bar(BA::Q_FULL + g), q_cnt[g] & 1, cx.abort_flag, p.status,
                         site + BA::Q_FULL + g) &&
               next_s(g, kv_cnt, 0, u.n[g]);
      for (int j = 0; ok && j < n_max; ++j) {
        const int t = kv_cnt + j;
        bool used = false;
#pragma unroll
        for (int g = g_lo; g <= g_hi; ++g) {
          const int n = u.n[g];
          if (!ok || j >= n) continue;
          used = true;
          // S_g(j+1) first: it only needs the softmax to have read S_g(j)
          ok = (j + 1 >= n || next_s(g, t + 1, j + 1, n)) && next_pv(g, t, j, n);
        }
        if (ok && !used) {
          // A tile none of this warp's query tiles uses: release its stage only
          // once it was loaded, so each release phase gets one arrival per MMA
          // warp (a warp running ahead would complete a phase on its own).
          ok = mbar_wait(cx.bar(BA::K_FULL + t % NS), (t / NS) & 1, cx.abort_flag, p.status,
                         site + BA::K_FULL + t % NS);
        }
        if (!ok) break;
        // the stage's K and V tiles are both done with (one release per stage)
        commit(BA::K_EMPTY + t % NS);
      }
      for (int g = 0; g < 2; ++g) q_cnt[g] += (u.n[g] > 0);
      kv_cnt += n_max;
    }
  } else {
    constexpr int g = GSEL;
    for (int k = 0; ok; ++k) {
      typename UnitSel<PAIRED>::T u;
      const int unit = next_unit<NS>(p, cx, k, kRoleMma, cx.lane == 0, u);
      if (unit < 0) break;
      const int n_slots = u.slots();
      if (n_slots == 0) continue;
      const int n = u.n[g];
      // prologue: S_g(0)
      if (n > 0)
        ok = mbar_wait(cx.bar(BA::Q_FULL + g), q_cnt[g] & 1, cx.abort_flag, p.status,
                       site + BA::Q_FULL + g) &&
             next_s(g, kv_cnt + u.slot_of(g, 0), 0, n);
      // Every slot of the unit, in load order: this warp's own key tiles get
      // S_g(j+1) (it only needs the softmax to have read S_g(j)) and then
      // PV_g(j); every slot, own or not, gets this warp's release.
      int j = 0;  // this warp's next key tile
      for (int slot = 0; ok && slot < n_slots; ++slot) {
        const int t = kv_cnt + slot;
        if (j < n && u.slot_of(g, j) == slot) {
          ok = (j + 1 >= n || next_s(g, kv_cnt + u.slot_of(g, j + 1), j + 1, n)) &&
               next_pv(g, t, j, n);
          ++j;
        } else {
          // A slot none of this warp's work uses: release it only once it was
          // loaded, so each release phase gets one arrival per MMA warp (a warp
          // running ahead would complete a phase on its own).
          ok = mbar_wait(cx.bar(BA::K_FULL + t % NS), (t / NS) & 1, cx.abort_flag, p.status,
                         site + BA::K_FULL + t % NS);
        }
        if (!ok) break;
        // the stage's K and V tiles are both done with (one release per stage)
        commit(BA::K_EMPTY + t % NS);
      }
      q_cnt[g] += (n > 0);
      kv_cnt += n_slots;
    }
  }
  // Every MMA this warp issued completes before TMEM is released.
  constexpr int dr = BA::DRAIN + (GSEL == 1 ? 1 : 0);
  commit(dr);
  volatile int never = 0;
  mbar_wait(cx.bar(dr), 0, &never, p.status, site + dr);
}

// Single MMA warp for both query tiles (P over S, d_k = 128): per key tile
// PV0(j), S0(j+1), PV1(j), S1(j+1), which keeps the two softmax warpgroups
// alternating on the tensor core.  (Measured: this fixed order is ~3 % faster
// here than two independent issuers.)
template <int D, bool NARROW>
__device__ __forceinline__ void mma_role_pair(const Bf16Params& p, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;
  static_assert(!C::SEPARATE_P && C::SPLIT_RELEASE, "pair order: P over S, split release");
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
  // the head's own widths when NARROW (as in mma_role)
  const int n_ks = NARROW ? p.dk_steps : D / 16;
  const uint32_t idesc_o =
      NARROW ? idesc_bf16_f32(128, p.dv_n, false, true) : idesc_bf16_f32(128, D, false, true);
  // K-major Q and K tiles: 8-row groups 1024 B apart; V MN-major with its
  // second 64-wide d chunk one CHUNK further.
  const uint64_t dq0 = smem_desc_sw128(cx.sQ, 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(cx.sK, 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(cx.sV, C::CHUNK, 1024);
  auto commit = [&](int id) {
    if (elect_one()) umma_commit(cx.bar(id));
    __syncwarp();
  };
  // S_g = Q_g K_t^T: M 128 queries, N 128 keys, K = d in steps of 16
  auto issue_s = [&](int g, int t) {
    const uint64_t a = dq0 + static_cast<uint64_t>((g * C::TILE) >> 4);
    const uint64_t b = dk0 + static_cast<uint64_t>(((t % NS) * C::TILE) >> 4);
    const uint32_t d_tmem = cx.tmem + (g ? C::TM_S1 : C::TM_S0);
    if (elect_one()) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        if (ks >= n_ks) break;
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ss(d_tmem, a + off, b + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(cx.bar(BA::S_FULL + g));
    }
    __syncwarp();
  };
  // O_g += P_g V_t: A = P_g from TMEM (16 keys = 8 columns per step),
  // B = V_t MN-major (16 keys = 16 rows of 128 B = 2048 B per step).
  auto issue_pv = [&](int g, int t, bool first) {
    const uint64_t b = dv0 + static_cast<uint64_t>(((t % NS) * C::TILE) >> 4);
    const uint32_t a_tmem = cx.tmem + (g ? C::TM_P1 : C::TM_P0);
    const uint32_t d_tmem = cx.tmem + (g ? C::TM_O1 : C::TM_O0);
    const uint32_t acc0 = first ? 0u : 1u;
    if (elect_one()) {
#pragma unroll
      for (int ks = 0; ks < kBlockN / 16; ++ks)
        umma_ts(d_tmem, a_tmem + 8u * ks, b + static_cast<uint64_t>((ks * 2048) >> 4), idesc_o,
                ks > 0 ? 1u : acc0);
    }
    __syncwarp();
  };
  int q_cnt[2] = {0, 0};  // units with Q_g so far
  int s_cnt[2] = {0, 0};  // P_g tiles consumed so far
  int s_iss[2] = {0, 0};  // S_g tiles issued so far
  int o_cnt[2] = {0, 0};  // units with O_g so far
  int kv_cnt = 0;
  bool ok = true;
  // S_g(t) for the unit's key tile j; with separate P the softmax must first
  // have read the previous S_g (any unit).  The last S_g of a unit frees Q_g.
  auto next_s = [&](int g, int t, int j, int n) {
    if constexpr (C::SEPARATE_P) {
      if (s_iss[g] > 0 && !mbar_wait(cx.bar(BA::S_FREE + g), (s_iss[g] - 1) & 1, cx.abort_flag,
                                     p.status, kRoleMma * 64 + BA::S_FREE + g))
        return false;
    }
    if (!mbar_wait(cx.bar(BA::K_FULL + t % NS), (t / NS) & 1, cx.abort_flag, p.status,
                   kRoleMma * 64 + BA::K_FULL + t % NS))
      return false;
    tc_fence_after();
    issue_s(g, t);
    ++s_iss[g];
    if (j + 1 == n) commit(BA::Q_FREE + g);
    return true;
  };
  // PV_g for key tile t (the unit's j-th); the unit's last PV_g releases O_g
  // to the epilogue.
  auto next_pv = [&](int g, int t, int j, int n) {
    const int s = t % NS;
    if (!mbar_wait(cx.bar(BA::P_FULL + g), s_cnt[g] & 1, cx.abort_flag, p.status,
                   kRoleMma * 64 + BA::P_FULL + g) ||
        !mbar_wait(cx.bar(BA::V_FULL + s), (t / NS) & 1, cx.abort_flag, p.status,
                   kRoleMma * 64 + BA::V_FULL + s))
      return false;
    // the previous unit's epilogue must have read O_g before it is overwritten
    if (j == 0 && o_cnt[g] > 0 &&
        !mbar_wait(cx.bar(BA::O_FREE + g), (o_cnt[g] - 1) & 1, cx.abort_flag, p.status,
                   kRoleMma * 64 + BA::O_FREE + g))
      return false;
    ++s_cnt[g];
    tc_fence_after();
    issue_pv(g, t, j == 0);
    if constexpr (C::SEPARATE_P) commit(BA::PV_DONE + g);
    if (j + 1 == n) {
      commit(BA::O_DONE + g);
      ++o_cnt[g];
    }
    return true;
  };
  for (int k = 0; ok; ++k) {
    typename UnitSel<false>::T u;
    const int unit = next_unit<NS>(p, cx, k, kRoleMma, cx.lane == 0, u);
    if (unit < 0) break;
    const int n_max = max(u.n[0], u.n[1]);
    if (n_max == 0) continue;
    // prologue: S0(0), S1(0); then K_0 is done with
    for (int g = 0; ok && g < 2; ++g) {
      if (u.n[g] == 0) continue;
      ok = mbar_wait(cx.bar(BA::Q_FULL + g), q_cnt[g] & 1, cx.abort_flag, p.status,
                     kRoleMma * 64 + BA::Q_FULL + g) &&
           next_s(g, kv_cnt, 0, u.n[g]);
    }
    if (ok) commit(BA::K_EMPTY + kv_cnt % NS);
    // Per key tile PV0(j), S0(j+1), PV1(j), S1(j+1).  V_j is released once
    // PV1(j) is done and K_{j+1} once S1(j+1) is, so a stage's next K load
    // starts a full key tile earlier than if both waited for the last MMA.
    for (int j = 0; ok && j < n_max; ++j) {
      const int t = kv_cnt + j;
      for (int g = 0; ok && g < 2; ++g) {
        if (j < u.n[g]) ok = next_pv(g, t, j, u.n[g]);
        if (ok && g == 1) commit(BA::V_EMPTY + t % NS);
        if (ok && j + 1 < u.n[g]) ok = next_s(g, t + 1, j + 1, u.n[g]);
      }
      if (ok && j + 1 < n_max) commit(BA::K_EMPTY + (t + 1) % NS);
    }
    for (int g = 0; g < 2; ++g) q_cnt[g] += (u.n[g] > 0);
    kv_cnt += n_max;
  }
  // Every MMA this warp issued completes before TMEM is released.
  commit(BA::DRAIN + 0);
  volatile int never = 0;
  mbar_wait(cx.bar(BA::DRAIN + 0), 0, &never, p.status, kRoleMma * 64 + BA::DRAIN);
}

// TOK: the two softmax warps on one sub-partition (the same lane quarter of Q0
// and Q1) take turns at the exponentials, passing a token through an mbarrier
// pair.  That keeps their SFU-bound phases apart, so each runs at the full SFU
// rate while the other does its loads, maxima and stores (d_k = 64 without the
// causal mask, where the SFU work per score equals the tensor work: +5 %).
template <int D, bool TOK, bool PAIRED, bool NARROW>
__device__ __forceinline__ void softmax_role(const Bf16Params& p, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  const int warp = cx.warp - kSoftmaxWarp0, lane = cx.lane;
  const int g = warp >> 2;                      // which query tile
  const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31 (= hardware warp % 4)
  const int row = quarter * 32 + lane;          // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = cx.tmem + (g ? C::TM_S1 : C::TM_S0) + lane_off;
  const uint32_t tP = cx.tmem + (g ? C::TM_P1 : C::TM_P0) + lane_off;
  const uint32_t tO = cx.tmem + (g ? C::TM_O1 : C::TM_O0) + lane_off;
  const uint32_t stage = cx.sStage + g * C::CHUNK;  // this warpgroup's staging chunk
  // one fixed thread issues, commits and waits for the TMA stores (bulk
  // async-groups belong to the issuing thread)
  const bool store_thread = (warp == 4 * g) && lane == 0;
  const float c2 = p.scale_log2;
  // O columns the P.V products write (d_v rounded up to 16; D unless NARROW)
  const int dv_n = NARROW ? p.dv_n : D;
  int s_cnt = 0;  // S_g tiles so far
  int o_cnt = 0;  // units with O_g so far
  int tok_cnt = 0;  // exponential turns taken so far
  // this warp's turn barrier and its partner's (same quarter, other tile)
  const int tok_wait = (g ? BA::TOK_B : BA::TOK_A) + quarter;
  const int tok_pass = (g ? BA::TOK_A : BA::TOK_B) + quarter;
  bool ok = true;
  for (int k = 0; ok; ++k) {
    // With the exponential turns the softmax decodes its unit itself
    // (measured: reading the scheduler's copy made those kernels 1-2 %
    // slower, while it makes the others 2-3 % faster).
    typename UnitSel<PAIRED>::T u;
    int unit;
    if constexpr (TOK) {
      UnitIndexOnly none;
      unit = next_unit<C::NS>(p, cx, k, kRoleSoftmax, lane == 0, none);
      if (unit >= 0) u = decode_unit<PAIRED>(p, unit);
    } else {
      unit = next_unit<C::NS>(p, cx, k, kRoleSoftmax, lane == 0, u);
    }
    if (unit < 0) break;
    const int q_start = u.qstart(g);
    const int qi = q_start + row;
    const int n_tiles = PAIRED ? (g ? u.n[1] : u.n[0]) : u.n[g];
    const int kv_len = u.keys(g);
    const int seq = u.seq(g);
    const int head = u.head(g);
    // Turns alternate Q0, Q1, Q0, ... over the key tiles both query tiles
    // have; Q1's warp hands Q0's the first turn of each unit.  Each side
    // passes only after it has waited for the other's pass, so no turn
    // barrier ever gets two phases ahead of its waiter.
    const int n_turns = TOK ? min(u.n[0], u.n[1]) : 0;
    if (g == 1 && n_turns > 0) mbar_arrive(cx.bar(tok_pass));
    float m_ref = 0.f;  // reference maximum (log2 units) the exponents use
    float l = 0.f;      // running sum of 2^(s*c2 - m_ref)
    for (int j = 0; j < n_tiles; ++j) {
      ok = mbar_wait(cx.bar(BA::S_FULL + g), s_cnt & 1, cx.abort_flag, p.status,
                     kRoleSoftmax * 64 + BA::S_FULL + g);
      if (!ok) break;
      ++s_cnt;
      tc_fence_after();
      uint32_t r[128];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        tmem_ld32(tS + 32u * c4, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c4]));
      tmem_ld_wait();
      if constexpr (C::SEPARATE_P) {
        // S_g has been read: the next S_g may be computed into it
        tc_fence_before();
        mbar_arrive(cx.bar(BA::S_FREE + g));
      }
      float x[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(r[c]);
      // per-element mask on the diagonal tile and a ragged last tile
      const int kbase = j * kBlockN;
      int lim = kv_len - kbase;                                    // keys c < lim exist
      if (masks_causal(p.mask_kind) && qi - kbase + 1 < lim) lim = qi - kbase + 1;
      if (lim < kBlockN) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) x[c] = -INFINITY;
      }
      // row maximum: eight independent chains of three-input max
      float mk[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mk[q] = fmaxf(x[2 * q], x[2 * q + 1]);
#pragma unroll
      for (int c = 16; c < 128; c += 16) {
#pragma unroll
        for (int q = 0; q < 8; ++q) mk[q] = fmax3(mk[q], x[c + 2 * q], x[c + 2 * q + 1]);
      }
      const float mx =
          fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7])) * c2;
      // Each row moves its own reference up to this tile's maximum when that
      // maximum exceeds it by more than the threshold; l and the partial
      // output are rescaled by alpha (rows that keep their reference use
      // exactly 1, so a row's arithmetic never depends on its neighbours).
      bool move = false;
      float alpha = 1.f;
      if (j == 0) {
        m_ref = (mx == -INFINITY) ? 0.f : mx;
      } else if (mx > m_ref + kRescaleThreshold) {
        move = true;
        alpha = ex2_approx(m_ref - mx);
        l *= alpha;
        m_ref = mx;
      }
      if (j < n_turns) {
        ok = mbar_wait(cx.bar(tok_wait), tok_cnt & 1, cx.abort_flag, p.status,
                       kRoleSoftmax * 64 + tok_wait);
        if (!ok) break;
        ++tok_cnt;
      }
      // p = 2^(s*c2 - m_ref): packed scale-subtract, ex2 on the SFU, packed sums
      const float nm = -m_ref;
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      // (each pair is packed to bf16 as soon as it exists, so the float32
      // values die at once and the row never holds 128 floats and 64 words)
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
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
      if (j < n_turns && (g == 0 || j + 1 < n_turns)) mbar_arrive(cx.bar(tok_pass));
      if constexpr (C::SEPARATE_P) {
        // PV_g of the previous tile must be done before P_g is rewritten and
        // O_g rescaled
        if (s_cnt > 1 && !mbar_wait(cx.bar(BA::PV_DONE + g), (s_cnt - 2) & 1, cx.abort_flag,
                                    p.status, kRoleSoftmax * 64 + BA::PV_DONE + g)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // P_g as bf16 pairs (A operand of P.V)
      tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tP + 32u, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      // (with P over S, PV_g(j-1) is complete already: S_g(j) was issued after it)
      if (__any_sync(0xffffffffu, move)) {
#pragma unroll
        for (int c32 = 0; c32 < D / 32; ++c32) {
          if (32 * c32 >= dv_n) break;  // O columns past d_v are never written
          uint32_t o[32];
          tmem_ld32(tO + 32u * c32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float a0, a1;
            mul2(a0, a1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha);
            o[i] = __float_as_uint(a0);
            o[i + 1] = __float_as_uint(a1);
          }
          tmem_st32(tO + 32u * c32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      // (test hook) withholding this CTA's first P leaves the MMA warp's
      // bounded wait to run out, which exercises the abort and drain path
      if (!(p.withhold_p && g == 0 && k == 0 && j == 0)) mbar_arrive(cx.bar(BA::P_FULL + g));
    }
    if (!ok) break;
    if (q_start >= p.Lq) continue;
    // ---- epilogue: O / l rounded to bf16, 64 columns at a time through this
    // warpgroup's staging chunk (128-byte swizzle) and a TMA store, which
    // skips rows past Lq.
    if (n_tiles > 0) {
      ok = mbar_wait(cx.bar(BA::O_DONE + g), o_cnt & 1, cx.abort_flag, p.status,
                     kRoleSoftmax * 64 + BA::O_DONE + g);
      if (!ok) break;
      tc_fence_after();
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    if (p.lse && qi < p.Lq) {
      // log of the softmax denominator, natural units: m_ref and the
      // exponents are in log2 units of the scaled scores
      p.lse[(static_cast<size_t>(seq) * p.H + head) * p.Lq + qi] =
          (l > 0.f) ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    // only the 64-column chunks that hold output columns (d_v <= 64 on the
    // 128-wide kernel stores one), and in them only the written 32-column
    // halves are read from TMEM
    const int n_chunks = (dv_n + 63) / 64;
#pragma unroll
    for (int c = 0; c < C::KCH; ++c) {
      if (c >= n_chunks) break;
      // the previous TMA store from the staging chunk must have read it
      if (store_thread) tma_store_wait_read();
      named_barrier(1 + g, 128);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        const bool written = 64 * c + 32 * half < dv_n;
        if (n_tiles > 0 && written) {
          tmem_ld32(tO + 64u * c + 32u * half, o);
          tmem_ld_wait();
          if (c == n_chunks - 1 && (half == 1 || 64 * c + 32 >= dv_n)) {
            // O_g may be overwritten by the next unit from here on
            tc_fence_before();
            mbar_arrive(cx.bar(BA::O_FREE + g));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[8 * v4 + 2 * i]) * inv,
                               __uint_as_float(o[8 * v4 + 2 * i + 1]) * inv);
          const uint32_t unit16 = static_cast<uint32_t>(4 * half + v4);  // 16-byte unit of the row
          const uint32_t addr = stage + row * 128 + ((unit16 ^ (row & 7)) << 4);
          st_shared_v4(addr, w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      named_barrier(1 + g, 128);
      if (store_thread) {
        tma_store_4d(&p.tm_o, stage, 64 * c, head, q_start, seq);
        tma_store_commit();
      }
      __syncwarp();
    }
    if (n_tiles > 0) ++o_cnt;
  }
  // the staging chunk must outlive the reads of the last store
  if (store_thread) tma_store_wait_read();
  __syncwarp();
}

template <int D, bool TOK, bool PAIRED, bool NARROW>
__global__ void __launch_bounds__(kThreads, 1) fwd_bf16_kernel(const __grid_constant__ Bf16Params p) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  Ctx cx;
  cx.sQ = s_base + C::OFF_Q;
  cx.sK = s_base + C::OFF_K;
  cx.sV = s_base + C::OFF_V;
  cx.sStage = s_base + C::OFF_STAGE;
  cx.s_bar = s_base + C::OFF_BAR;
  cx.warp = static_cast<int>(threadIdx.x >> 5);
  cx.lane = static_cast<int>(threadIdx.x & 31);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  cx.abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  cx.unit_slot = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  cx.unit_data = reinterpret_cast<volatile int*>(smem + C::OFF_UNITS);
  cx.clc_resp = s_base + C::OFF_CLC;

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int g = 0; g < 2; ++g) {
      mbar_init(cx.bar(BA::Q_FULL + g), 1);
      mbar_init(cx.bar(BA::Q_FREE + g), 1);
      mbar_init(cx.bar(BA::S_FULL + g), 1);
      mbar_init(cx.bar(BA::P_FULL + g), 128);
      mbar_init(cx.bar(BA::O_DONE + g), 1);
      mbar_init(cx.bar(BA::O_FREE + g), 128);
      mbar_init(cx.bar(BA::UNIT_FULL + g), 1);
      mbar_init(cx.bar(BA::UNIT_EMPTY + g), unit_consumers<D>());
      mbar_init(cx.bar(BA::S_FREE + g), 128);
      mbar_init(cx.bar(BA::PV_DONE + g), 1);
    }
    mbar_init(cx.bar(BA::CLC), 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(cx.bar(BA::TOK_A + q), 32);
      mbar_init(cx.bar(BA::TOK_B + q), 32);
    }
    mbar_init(cx.bar(BA::DRAIN + 0), 1);
    mbar_init(cx.bar(BA::DRAIN + 1), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(cx.bar(BA::K_FULL + s), 1);
      mbar_init(cx.bar(BA::V_FULL + s), 1);
      mbar_init(cx.bar(BA::K_EMPTY + s), C::SEPARATE_P ? 2 : 1);
      mbar_init(cx.bar(BA::V_EMPTY + s), 1);
    }
    *cx.abort_flag = 0;
    fence_mbar_init();
  }
  if (cx.warp == kProducerWarp && cx.lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_o);
  }
  if (cx.warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  // The set-up above touches no global memory, so it may overlap the end of
  // the previous kernel on the stream; everything below comes after it.  (No
  // early trigger for the next launch: its CTAs start as this grid's CTAs
  // exit.  Measured: triggering at the start of each CTA made the persistent
  // grids 5-12 % slower, at the end of each CTA the causal base decoder 5 %
  // slower; this way one-wave grids gain 0.3-0.4 us and the rest is unchanged.)
  griddep_wait();

  if (cx.warp < kSoftmaxWarp0 + 8) {
    regs_increase<C::REGS_SOFTMAX>();
    softmax_role<D, TOK, PAIRED, NARROW>(p, cx);
  } else {
    regs_decrease<C::REGS_OTHER>();
    if (cx.warp == kMmaWarp) {
      if constexpr (C::SEPARATE_P) {
        mma_role<D, 0, PAIRED, NARROW>(p, cx);
      } else {
        mma_role_pair<D, NARROW>(p, cx);
      }
    } else if (cx.warp == kMma1Warp) {
      if constexpr (C::SEPARATE_P) mma_role<D, 1, PAIRED, NARROW>(p, cx);
    } else if (cx.warp == kProducerWarp) {
      if constexpr (PAIRED) {
        producer_role_paired<D>(p, cx);
      } else {
        producer_role<D>(p, cx);
      }
    } else {
      scheduler_role<D, PAIRED>(p, cx);
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (cx.warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, C::TMEM_COLS);
  }
}

template <int D, bool TOK, bool PAIRED, bool NARROW>
cudaError_t launch_d(const Bf16Params& p, cudaStream_t stream, LaunchInfo* info) {
  static_assert(!PAIRED || D == 64, "heads are paired only with one MMA warp per query tile");
  static_assert(!(TOK && NARROW), "the narrow instantiations take no exponential turns");
  using C = Cfg<D>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};  // the attribute is per device and function
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(fwd_bf16_kernel<D, TOK, PAIRED, NARROW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long units = static_cast<long long>(p.n_qtiles) *
                          (PAIRED ? (static_cast<long long>(p.B) * p.H + 1) / 2
                                  : static_cast<long long>(p.B) * p.H);
  const dim3 grid(static_cast<unsigned>(units));
  e = launch_serialized(fwd_bf16_kernel<D, TOK, PAIRED, NARROW>, grid, dim3(kThreads), C::SMEM, stream, p);
  if (e != cudaSuccess) return e;
  if (info) {
    info->kernels = 1;
    info->grid = static_cast<int>(units);
    info->block = kThreads;
    info->smem = C::SMEM;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const Bf16Params& params, int d, cudaStream_t stream,
                            LaunchInfo* info) {
  Bf16Params p = params;
  {
    // K and V bytes of one head (d_k-wide keys, the kernel's width for values)
    const long long per_head = 2ll * p.Lk * d * 2 > 0 ? 2ll * p.Lk * d * 2 : 1;
    long long hg = kHeadGroupBytes / per_head;
    const long long bh = static_cast<long long>(p.B) * p.H;
    if (hg > bh) hg = bh;
    if (hg < 2) hg = 2;
    p.head_group = static_cast<int>(hg) & ~1;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  // Pairing heads (d_k = 64 only, where each query tile has its own MMA
  // warp).  With a single query tile per head a shared unit leaves its second
  // tile, and half of the softmax warps, idle; pairing halves the units and
  // runs two heads per SM at once, which pays when the shared units would
  // take more than one wave of the SMs (measured: 256 heads of 128 rows
  // 9.1 -> 7.4 us; 128 heads of one query row against 4096 keys 33 -> 57 us,
  // where pairing leaves half of the SMs idle).  With two or more query tiles
  // per head, sharing each K/V tile between them is faster.
  p.paired = (d == 64 && p.Lq <= kBlockM && static_cast<long long>(p.B) * p.H > sms) ? 1 : 0;
  if (p.paired) {
    const long long units = static_cast<long long>((p.Lq + kBlockM - 1) / kBlockM) *
                            ((static_cast<long long>(p.B) * p.H + 1) / 2);
    if (units > 0x7fffffffll) return cudaErrorInvalidValue;
    p.n_qtiles = (p.Lq + kBlockM - 1) / kBlockM;
  }
  // (the exponential turn-taking pays off at d_k = 64 without the causal
  // mask once units span several key tiles; with one or two key tiles the
  // hand-over at the start of each unit costs more than it saves)
  // A head narrower than the kernel (d_k or d_v below 64 or 128) runs an
  // instantiation that issues only its own K steps and output columns; the
  // full-width ones keep those counts as compile-time constants.
  const bool narrow = p.dk_steps * 16 < d || p.dv_n < d;
  if (d == 64) {
    if (narrow)
      return p.paired ? launch_d<64, false, true, true>(p, stream, info)
                      : launch_d<64, false, false, true>(p, stream, info);
    const bool tok = !masks_causal(p.mask_kind) && p.Lk >= 4 * kBlockN;
    if (p.paired)
      return tok ? launch_d<64, true, true, false>(p, stream, info)
                 : launch_d<64, false, true, false>(p, stream, info);
    return tok ? launch_d<64, true, false, false>(p, stream, info)
               : launch_d<64, false, false, false>(p, stream, info);
  }
  if (d == 128)
    return narrow ? launch_d<128, false, false, true>(p, stream, info)
                  : launch_d<128, false, false, false>(p, stream, info);
  return cudaErrorInvalidValue;
}

}  // namespace mha
