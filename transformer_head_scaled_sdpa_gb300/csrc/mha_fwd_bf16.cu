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
// One CTA = one work unit: (b, h, two 128-row query tiles Q0, Q1) sharing
// every K/V tile.  384 threads (three warpgroups) in four roles:
//   warps 0-3   softmax for Q0 (thread r owns row r = TMEM lane r)
//   warps 4-7   softmax for Q1
//   warp 8      TMEM allocator and MMA issuer (one thread)
//   warp 9      TMA producer: Q0, Q1, then K_j / V_j into an NS-stage ring
//   warps 10-11 idle
// The third warpgroup gives registers to the softmax warpgroups, which hold
// a whole 128-score row per thread: launched at 168 per thread, it drops to
// 64 (d_k 64) or 80 (d_k 128) and they rise to 216 or 208 (both splits total
// 63488 <= 384*168 registers).
// TMEM (512 columns): S0 | S1 | O0 | O1.  Softmax g reads S_g (float32),
// writes P_g as bf16 pairs into the first 64 columns of S_g, and the P.V
// MMA reads P_g from TMEM.  Per key tile j the MMA warp issues
//   PV0(j), S0(j+1), PV1(j), S1(j+1)
// so softmax 0 works on S0(j+1) while the tensor core runs PV1(j) and
// S1(j+1), and vice versa.  MMAs of one thread run in issue order, so
// S_g(j+1) overwrites P_g(j) only after PV_g(j) has read it, and once S_g(j+1)
// is complete PV_g(j) is too: softmax g may rescale O_g in place then.
// Masks: causal tiles above the diagonal are never loaded or computed; the
// diagonal tile and a ragged last key tile are masked per element (score set
// to -inf, weight exactly 0: formula page, 応用, 先を読まない仕掛け).
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p stays <= 2^8
constexpr int kHeadGroup = 32;              // heads dispatched together (L2 reuse of K/V)

template <int D>
struct Cfg {
  static constexpr int KCH = D / 64;             // 128-byte chunks along d
  static constexpr int CHUNK = 128 * 128;        // one [128 rows x 128 B] swizzled chunk
  static constexpr int TILE = KCH * CHUNK;       // one 128-row Q, K or V tile
  static constexpr int NS = (D == 64) ? 4 : 2;   // K/V ring stages
  static constexpr int OFF_Q = 0;                // Q0, Q1
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  static constexpr int NBAR = 9 + 3 * NS;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  // TMEM columns
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128;
  static constexpr uint32_t TM_O0 = 256, TM_O1 = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  // registers per thread after rebalancing (softmax warpgroups, the rest)
  static constexpr uint32_t REGS_SOFTMAX = (D == 64) ? 216 : 208;
  static constexpr uint32_t REGS_OTHER = (D == 64) ? 64 : 80;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(256 * REGS_SOFTMAX + 128 * REGS_OTHER <= kThreads * 168, "register split");
};

// barrier ids inside the barrier block
template <int NS>
struct Bars {
  static constexpr int Q_FULL = 0;                // + g
  static constexpr int S_FULL = 2;                // + g
  static constexpr int P_FULL = 4;                // + g
  static constexpr int O_DONE = 6;                // + g
  static constexpr int DRAIN = 8;
  static constexpr int K_FULL = 9;                // + stage
  static constexpr int V_FULL = 9 + NS;           // + stage
  static constexpr int KV_EMPTY = 9 + 2 * NS;     // + stage
};

// role ids for the status "site" field
constexpr int kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3;

struct Unit {
  int b, h;
  int q0;       // first query row of Q0
  int n[2];     // key tiles for Q0, Q1
  int kv_len;   // keys visible before the causal limit
};

__device__ __forceinline__ Unit decode_unit(const Bf16Params& p, int unit) {
  // Units are dispatched in groups of kHeadGroup heads, so a group's K/V stay
  // in L2 while all of its query blocks run; inside a group the causal blocks
  // go heaviest first.
  const int bh_count = p.B * p.H;
  const int n_pairs = p.n_qtiles;  // query blocks of 256 rows
  const int group = unit / (kHeadGroup * n_pairs);
  const int within = unit - group * kHeadGroup * n_pairs;
  const int heads_here = min(kHeadGroup, bh_count - group * kHeadGroup);
  const int pair_idx = within / heads_here;
  const int bh = group * kHeadGroup + within % heads_here;
  const int t = (p.mask_kind == kMaskCausal) ? (n_pairs - 1 - pair_idx) : pair_idx;
  Unit u;
  u.b = bh / p.H;
  u.h = bh % p.H;
  u.q0 = t * kUnitRows;
  int kv_len = p.Lk;
  if (p.mask_kind == kMaskKeyPadding) {
    const int len = __ldg(p.key_lens + u.b);
    kv_len = len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
  }
  u.kv_len = kv_len;
  const int n_kv = (kv_len + kBlockN - 1) / kBlockN;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int qs = u.q0 + g * kBlockM;
    int n = (qs < p.Lq) ? n_kv : 0;
    if (p.mask_kind == kMaskCausal && n > qs / kBlockN + 1) n = qs / kBlockN + 1;
    u.n[g] = n;
  }
  return u;
}

// Per-CTA context shared by the roles.
struct Ctx {
  uint32_t sQ, sK, sV, s_bar;
  uint32_t tmem;
  volatile int* abort_flag;
  int warp, lane;
  __device__ __forceinline__ uint32_t bar(int id) const {
    return s_bar + 8u * static_cast<uint32_t>(id);
  }
};

// TMA producer (warp 9): Q0, K_0, Q1, V_0, then K_j / V_j into the ring.
// The whole warp runs the loop and waits; one elected lane issues.
template <int D>
__device__ __forceinline__ void producer_role(const Bf16Params& p, const Unit& u, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;
  const int n_max = max(u.n[0], u.n[1]);
  if (n_max == 0) return;
  auto load_q = [&](int g) {
    if (elect_one()) {
      mbar_arrive_expect_tx(cx.bar(BA::Q_FULL + g), C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d(cx.sQ + g * C::TILE + c * C::CHUNK, &p.tm_q, cx.bar(BA::Q_FULL + g), 64 * c,
                    u.h, u.q0 + g * kBlockM, u.b);
    }
    __syncwarp();
  };
  auto load_kv = [&](int j, bool is_v) {
    const int s = j % NS;
    const uint32_t dst = (is_v ? cx.sV : cx.sK) + s * C::TILE;
    const uint32_t full = cx.bar((is_v ? BA::V_FULL : BA::K_FULL) + s);
    if (elect_one()) {
      mbar_arrive_expect_tx(full, C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d(dst + c * C::CHUNK, is_v ? &p.tm_v : &p.tm_k, full, 64 * c, u.h,
                    j * kBlockN, u.b);
    }
    __syncwarp();
  };
  if (u.n[0] > 0) load_q(0);
  load_kv(0, false);
  if (u.n[1] > 0) load_q(1);
  load_kv(0, true);
  int last = 0;  // last tile issued
  for (int j = 1; j < n_max; ++j) {
    const int s = j % NS;
    if (j >= NS) {
      if (!mbar_wait(cx.bar(BA::KV_EMPTY + s), ((j / NS) - 1) & 1, cx.abort_flag, p.status,
                     kRoleProducer * 64 + BA::KV_EMPTY + s))
        break;
    }
    load_kv(j, false);
    load_kv(j, true);
    last = j;
  }
  // Leave only when every copy this warp started has landed (the normal
  // path finds them complete already): the last load into each used stage.
  for (int g = 0; g < 2; ++g)
    if (u.n[g] > 0)
      mbar_wait(cx.bar(BA::Q_FULL + g), 0, cx.abort_flag, p.status, kRoleProducer * 64 + BA::Q_FULL);
  for (int j = (last + 1 > NS ? last + 1 - NS : 0); j <= last; ++j) {
    const int s = j % NS;
    mbar_wait(cx.bar(BA::K_FULL + s), (j / NS) & 1, cx.abort_flag, p.status,
              kRoleProducer * 64 + BA::K_FULL + s);
    mbar_wait(cx.bar(BA::V_FULL + s), (j / NS) & 1, cx.abort_flag, p.status,
              kRoleProducer * 64 + BA::V_FULL + s);
  }
}

// MMA issuer (warp 8): the whole warp runs the loop and the waits; one
// elected lane issues every tcgen05.mma and tcgen05.commit, with
// descriptors built once and stepped by compile-time offsets.
template <int D>
__device__ __forceinline__ void mma_role(const Bf16Params& p, const Unit& u, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;
  const int n_max = max(u.n[0], u.n[1]);
  if (n_max == 0) return;
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
  // K-major Q and K tiles: 8-row groups 1024 B apart; V MN-major with its
  // second 64-wide d chunk one CHUNK further.
  const uint64_t dq0 = smem_desc_sw128(cx.sQ, 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(cx.sK, 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(cx.sV, C::CHUNK, 1024);
  // S_g = Q_g K_j^T: M 128 queries, N 128 keys, K = d in steps of 16
  auto issue_s = [&](int g, int j) {
    const uint64_t a = dq0 + static_cast<uint64_t>((g * C::TILE) >> 4);
    const uint64_t b = dk0 + static_cast<uint64_t>(((j % NS) * C::TILE) >> 4);
    const uint32_t d_tmem = cx.tmem + (g ? C::TM_S1 : C::TM_S0);
    if (elect_one()) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ss(d_tmem, a + off, b + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(cx.bar(BA::S_FULL + g));
    }
    __syncwarp();
  };
  // O_g += P_g V_j: A = P_g from TMEM (16 keys = 8 columns per step),
  // B = V_j MN-major (16 keys = 16 rows of 128 B = 2048 B per step).
  auto issue_pv = [&](int g, int j) {
    const uint64_t b = dv0 + static_cast<uint64_t>(((j % NS) * C::TILE) >> 4);
    const uint32_t a_tmem = cx.tmem + (g ? C::TM_S1 : C::TM_S0);
    const uint32_t d_tmem = cx.tmem + (g ? C::TM_O1 : C::TM_O0);
    const uint32_t acc0 = j > 0 ? 1u : 0u;
    if (elect_one()) {
#pragma unroll
      for (int ks = 0; ks < kBlockN / 16; ++ks)
        umma_ts(d_tmem, a_tmem + 8u * ks, b + static_cast<uint64_t>((ks * 2048) >> 4), idesc_o,
                ks > 0 ? 1u : acc0);
    }
    __syncwarp();
  };
  auto commit = [&](int id) {
    if (elect_one()) umma_commit(cx.bar(id));
    __syncwarp();
  };
  bool ok = mbar_wait(cx.bar(BA::K_FULL), 0, cx.abort_flag, p.status, kRoleMma * 64 + BA::K_FULL);
  // prologue: S0(0), S1(0)
  for (int g = 0; ok && g < 2; ++g) {
    if (u.n[g] == 0) continue;
    ok = mbar_wait(cx.bar(BA::Q_FULL + g), 0, cx.abort_flag, p.status, kRoleMma * 64 + BA::Q_FULL);
    if (!ok) break;
    tc_fence_after();
    issue_s(g, 0);
  }
  for (int j = 0; ok && j < n_max; ++j) {
    const int s = j % NS;
    const uint32_t ph = (j / NS) & 1;
    for (int g = 0; g < 2; ++g) {
      if (j >= u.n[g]) continue;
      ok = mbar_wait(cx.bar(BA::P_FULL + g), j & 1, cx.abort_flag, p.status,
                     kRoleMma * 64 + BA::P_FULL + g) &&
           mbar_wait(cx.bar(BA::V_FULL + s), ph, cx.abort_flag, p.status,
                     kRoleMma * 64 + BA::V_FULL + s);
      if (!ok) break;
      tc_fence_after();
      issue_pv(g, j);
      if (j + 1 < u.n[g]) {
        const int s1 = (j + 1) % NS;
        ok = mbar_wait(cx.bar(BA::K_FULL + s1), ((j + 1) / NS) & 1, cx.abort_flag, p.status,
                       kRoleMma * 64 + BA::K_FULL + s1);
        if (!ok) break;
        tc_fence_after();
        issue_s(g, j + 1);
      } else {
        commit(BA::O_DONE + g);
      }
    }
    if (!ok) break;
    commit(BA::KV_EMPTY + s);
  }
  // Every MMA this warp issued completes before TMEM is released.
  commit(BA::DRAIN);
  volatile int never = 0;
  mbar_wait(cx.bar(BA::DRAIN), 0, &never, p.status, kRoleMma * 64 + BA::DRAIN);
}

template <int D>
__device__ __forceinline__ void softmax_role(const Bf16Params& p, const Unit& u, const Ctx& cx) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  const int warp = cx.warp, lane = cx.lane;
  const uint32_t tmem = cx.tmem;
  volatile int* abort_flag = cx.abort_flag;
  auto bar = [&](int id) { return cx.bar(id); };
  const int g = warp >> 2;                      // which query tile
  const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
  const int row = quarter * 32 + lane;          // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + (g ? C::TM_S1 : C::TM_S0) + lane_off;
  const uint32_t tO = tmem + (g ? C::TM_O1 : C::TM_O0) + lane_off;
  const float c2 = p.scale_log2;
  const int q_start = u.q0 + g * kBlockM;
  const int qi = q_start + row;
  const int n_tiles = u.n[g];
  float m_ref = 0.f;  // reference maximum (log2 units) the exponents use
  float l = 0.f;      // running sum of 2^(s*c2 - m_ref)
  bool ok = true;
  for (int j = 0; j < n_tiles; ++j) {
    ok = mbar_wait(bar(BA::S_FULL + g), j & 1, abort_flag, p.status,
                   kRoleSoftmax * 64 + BA::S_FULL + g);
    if (!ok) break;
    tc_fence_after();
    uint32_t r[128];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      tmem_ld32(tS + 32u * c4, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c4]));
    tmem_ld_wait();
    float x[128];
#pragma unroll
    for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(r[c]);
    // per-element mask on the diagonal tile and a ragged last tile
    const int kbase = j * kBlockN;
    int lim = u.kv_len - kbase;                                  // keys c < lim exist
    if (p.mask_kind == kMaskCausal && qi - kbase + 1 < lim) lim = qi - kbase + 1;
    if (lim < kBlockN) {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c >= lim) x[c] = -INFINITY;
    }
    // row maximum: eight independent chains of three-input max
    float mk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mk[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
    for (int c = 16; c < 128; c += 16) {
#pragma unroll
      for (int k = 0; k < 8; ++k) mk[k] = fmax3(mk[k], x[c + 2 * k], x[c + 2 * k + 1]);
    }
    const float mx =
        fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7])) * c2;
    if (j == 0) {
      m_ref = (mx == -INFINITY) ? 0.f : mx;
    } else {
      // Each row moves its own reference up to this tile's maximum when that
      // maximum exceeds it by more than the threshold; the partial output is
      // rescaled in place (PV_g(j-1) is complete: S_g(j) was issued after
      // it).  Rows that keep their reference multiply by exactly 1, so a
      // row's arithmetic never depends on its neighbours.
      const bool move = mx > m_ref + kRescaleThreshold;
      const float alpha = move ? ex2_approx(m_ref - mx) : 1.f;
      if (move) {
        l *= alpha;
        m_ref = mx;
      }
      if (__any_sync(0xffffffffu, move)) {
#pragma unroll
        for (int c32 = 0; c32 < D / 32; ++c32) {
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
    }
    // p = 2^(s*c2 - m_ref): packed scale-subtract, ex2 on the SFU, packed sums
    const float nm = -m_ref;
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 128; c += 2) {
      fma2(x[c], x[c + 1], x[c], x[c + 1], c2, c2, nm, nm);
      x[c] = ex2_approx(x[c]);
      x[c + 1] = ex2_approx(x[c + 1]);
      const int k = (c >> 1) & 3;
      add2(sa[k], sb[k], sa[k], sb[k], x[c], x[c + 1]);
    }
    add2(sa[0], sb[0], sa[0], sb[0], sa[1], sb[1]);
    add2(sa[2], sb[2], sa[2], sb[2], sa[3], sb[3]);
    l += (sa[0] + sb[0]) + (sa[2] + sb[2]);
    // P_g as bf16 pairs into the first 64 columns of S_g (A operand of P.V)
    uint32_t pk[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) pk[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
    tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
    tmem_st32(tS + 32u, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
    tmem_st_wait();
    tc_fence_before();
    // (test hook) withholding the first P of tile 0 leaves the MMA warp's
    // bounded wait to run out, which exercises the abort and drain path
    if (!(p.withhold_p && g == 0 && j == 0)) mbar_arrive(bar(BA::P_FULL + g));
  }
  if (ok && n_tiles > 0) {
    ok = mbar_wait(bar(BA::O_DONE + g), 0, abort_flag, p.status,
                   kRoleSoftmax * 64 + BA::O_DONE + g);
    tc_fence_after();
  }
  if (ok && q_start < p.Lq) {
    // epilogue: O / l rounded to bf16, staged in shared memory (the Q_g tile
    // buffer: every S_g MMA is complete) in the 128-byte-swizzled layout and
    // written by TMA stores, which skip rows past Lq.
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    const uint32_t stage = cx.sQ + g * C::TILE;
#pragma unroll
    for (int c32 = 0; c32 < D / 32; ++c32) {
      uint32_t o[32];
      if (n_tiles > 0) {
        tmem_ld32(tO + 32u * c32, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
      // 32 columns = 64 bytes = four 16-byte units of the 128-byte row
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) {
        const uint32_t unit = static_cast<uint32_t>((c32 & 1) * 4 + v4);
        const uint32_t addr = stage + (c32 >> 1) * C::CHUNK + row * 128 + ((unit ^ (row & 7)) << 4);
        st_shared_v4(addr, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
      }
    }
    fence_proxy_async_smem();
    named_barrier(1 + g, 128);
    if (warp == 4 * g && elect_one()) {
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) tma_store_4d(&p.tm_o, stage + c * C::CHUNK, 64 * c, u.h, q_start, u.b);
      tma_store_commit();
      tma_store_wait_read();  // the staging buffer must outlive the reads
    }
    __syncwarp();
  }
}

template <int D>
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
  cx.s_bar = s_base + C::OFF_BAR;
  cx.warp = static_cast<int>(threadIdx.x >> 5);
  cx.lane = static_cast<int>(threadIdx.x & 31);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  cx.abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Unit u = decode_unit(p, static_cast<int>(blockIdx.x));

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int g = 0; g < 2; ++g) {
      mbar_init(cx.bar(BA::Q_FULL + g), 1);
      mbar_init(cx.bar(BA::S_FULL + g), 1);
      mbar_init(cx.bar(BA::P_FULL + g), 128);
      mbar_init(cx.bar(BA::O_DONE + g), 1);
    }
    mbar_init(cx.bar(BA::DRAIN), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(cx.bar(BA::K_FULL + s), 1);
      mbar_init(cx.bar(BA::V_FULL + s), 1);
      mbar_init(cx.bar(BA::KV_EMPTY + s), 1);
    }
    *cx.abort_flag = 0;
    fence_mbar_init();
  }
  if (cx.warp == 9 && cx.lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (cx.warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;

  if (cx.warp < 8) {
    regs_increase<C::REGS_SOFTMAX>();
    softmax_role<D>(p, u, cx);
  } else {
    regs_decrease<C::REGS_OTHER>();
    if (cx.warp == 8) {
      mma_role<D>(p, u, cx);
    } else if (cx.warp == 9) {
      producer_role<D>(p, u, cx);
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (cx.warp == 8) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const Bf16Params& p, cudaStream_t stream, LaunchInfo* info) {
  using C = Cfg<D>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};  // the attribute is per device and function
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long units = static_cast<long long>(p.n_qtiles) * p.B * p.H;
  const dim3 grid(static_cast<unsigned>(units));
  fwd_bf16_kernel<D><<<grid, kThreads, C::SMEM, stream>>>(p);
  if (info) {
    info->kernels = 1;
    info->grid = static_cast<int>(units);
    info->block = kThreads;
    info->smem = C::SMEM;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const Bf16Params& p, int d, cudaStream_t stream, LaunchInfo* info) {
  if (d == 64) return launch_d<64>(p, stream, info);
  if (d == 128) return launch_d<128>(p, stream, info);
  return cudaErrorInvalidValue;
}

}  // namespace mha
