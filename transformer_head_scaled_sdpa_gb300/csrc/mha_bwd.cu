// mha_bwd.cu -- gradient of the bf16 attention forward (dQ, dK, dV), sm_103a.
//
// For a loss L with dL/dO given, every row i of (b, h) has weights
// a_ij = exp(s_ij - lse_i) (s = scale * q . k over its visible keys, lse the
// forward's row log-sum-exp) and, with g_ij = dO_i . v_j, the formula page's
// derivative of the weights by the scores (transformer-attention, section 証明:
// da_j/ds_i = a_j (delta_ij - a_i)) gives
//   dS_ij = a_ij (g_ij - D_i),   D_i = sum_j a_ij g_ij = dO_i . O_i
//   dV_j  = sum_i a_ij dO_i,     dK_j = scale sum_i dS_ij q_i,
//   dQ_i  = scale sum_j dS_ij k_j.
// Two kernels, in this order on the stream:
//   bwd_dq_kernel     units (b, h, 128-query tile); first forms D_i for
//                     its rows (stored for the next kernel) and copies the
//                     unit's Q and dO into TMEM, then the key tiles it sees
//                     stream through a two-stage ring: S = Q K^T and
//                     dP = dO V^T (A operands from TMEM), then dS (bf16, over
//                     S), then dQ += dS K.
//   bwd_dkdv_kernel   units (b, h, 128-key tile); the query tiles that
//                     see the keys stream through a two-stage ring.  Per query
//                     tile: S^T = K Q^T and dP^T = V dO^T on the tensor cores
//                     (keys on TMEM lanes), the sixteen gradient warps turn them
//                     into P^T and dS^T (bf16, written over S^T and dP^T in
//                     TMEM), and dV += P^T dO, dK += dS^T Q accumulate in TMEM
//                     (A operands from TMEM).
// Both take each streamed tile in two halves of 64 rows with TMEM regions of
// their own: the tensor cores run one half's products (and the next tile's
// scores) while the gradient warps turn the other half's scores into P, dS.
// Both are persistent: one CTA per SM runs unit after unit (cluster launch
// control), loading the next unit's fixed tiles and issuing its first scores
// while the current unit's epilogue drains (the dQ kernel loads them a unit
// ahead: once copied into TMEM, its Q and dO are not read from shared memory).
// Every operand reuses the forward's shared-memory layout (128-row tiles of
// 64-feature, 128-byte swizzled chunks): K-major as an operand whose
// reduction runs over d, MN-major where it runs over the rows.
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

constexpr int kBwdThreads = 608;  // warps 0-15 gradient, 16 MMA, 17 TMA, 18 scheduler
constexpr int kGradThreads = 512;
constexpr int kMmaWarp = 16, kTmaWarp = 17, kSchedWarp = 18;
// unit-queue readers: 16 gradient warps, the MMA warp, the TMA lane
constexpr int kBwdUnitConsumers = 18;
constexpr int kRoleBwdProducer = 8, kRoleBwdMma = 9, kRoleBwdGrad = 10, kRoleBwdSched = 11;

template <int D>
struct BwdCfg {
  static constexpr int KCH = D / 64;
  static constexpr int CHUNK = 128 * 128;
  static constexpr int TILE = KCH * CHUNK;     // one 128-row operand tile
  // fixed tiles A0, A1 (K, V or Q, dO) and a two-stage ring of tile pairs
  static constexpr int OFF_A0 = 0;
  static constexpr int OFF_A1 = TILE;
  static constexpr int OFF_RING = 2 * TILE;    // stage s: pair at OFF_RING + s * 2 * TILE
  static constexpr int OFF_VEC = OFF_RING + 4 * TILE;  // dQ kernel: D halves [2][128]
  static constexpr int OFF_BAR = OFF_VEC + 2 * 128 * 4;
  static constexpr int NBAR = 22;
  // tmem slot (+0), abort flag (+4), unit queue (+8, +12), cancellation
  // response (+16, 16 bytes, 16-byte aligned)
  static constexpr int OFF_MISC = (OFF_BAR + 8 * NBAR + 15) / 16 * 16;
  // the dQ kernel also stages the forward output O (for D = dO . O)
  static constexpr int OFF_O = (OFF_MISC + 32 + 1023) / 1024 * 1024;
  static constexpr int SMEM_DQ = OFF_O + TILE + 1024;
  static_assert(SMEM_DQ <= 227 * 1024, "shared memory budget (dQ)");
  // the dK/dV kernel stages one 64-column chunk of dV and of dK there for
  // its TMA stores
  static constexpr int OFF_STG = OFF_O;
  static constexpr int SMEM_DKDV = OFF_STG + 2 * CHUNK + 1024;
  static_assert(SMEM_DKDV <= 227 * 1024, "shared memory budget (dK/dV)");
  // TMEM: a tile's score-shaped matrices in two halves of 64 columns, half
  // hf at columns 128 hf (S or S^T) and 128 hf + 64 (dP or dP^T); then the
  // d-wide accumulators
  static constexpr uint32_t TM_HALF = 128, TM_DP = 64, TM_ACC0 = 256, TM_ACC1 = 256 + D;
  // the dQ kernel: its unit's Q and dO as bf16 pairs (A operands of the
  // score products) after the dQ accumulator
  static constexpr uint32_t TM_QA = 256 + D, TM_DOA = 256 + D + D / 2;
  static constexpr uint32_t TMEM_COLS = 512;
};

// barrier ids.  kScores + hf: the score products of half hf are in TMEM;
// kGrads + hf: the gradient warps have written P and dS of half hf.
enum { kFixFull = 0, kRingFull = 1, kRingEmpty = 3, kScores = 5, kGrads = 7, kAccDone = 9,
       kDrain = 10,
       // the persistent dK/dV kernel: the unit's last score products are done
       // with K and V; the epilogue has read the accumulators; the unit queue
       kFixFree = 11, kAccFree = 12, kUnitFull = 13, kUnitEmpty = 15, kClc = 17,
       // the dQ kernel: the gradient warps have read the unit's staged Q, dO
       // and O tiles (D formed, Q and dO copied into TMEM)
       kOFree = 18,
       // the dK/dV epilogue: a chunk is staged (512 arrivals); its TMA stores
       // have read the staging buffers
       kStgFull = 19, kStgFree = 20,
       // the dQ kernel: the unit's Q and dO are in TMEM (copied by the
       // gradient warps)
       kQTmem = 21 };

// TMEM column of the 16 rows of K16 step ks (0..3) of a half, packed as bf16
// pairs: they are chunk ks (one gradient warp's 16 columns), kept in its
// first 8 columns
__device__ __forceinline__ constexpr uint32_t a_col(int ks) { return 16u * static_cast<uint32_t>(ks); }

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// bf16 halves of a packed pair -> float (exact)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// CTA order: groups of p.head_group heads, so the tiles a group's CTAs all
// stream (Q and dO, or K and V) stay in L2 while the group runs; inside a group
// the tile index t runs over all of the group's heads before moving on, which
// puts the heavy causal tiles of every head first and leaves the grid a light
// tail.  Returns t (0 = the first launched) and sets *bh.
// The group holds about kBwdHeadGroupBytes of the streamed tiles (measured:
// 32 heads suit the GPT-3-like gradient and 64 big16 L 2048, 1 MiB and
// 512 KiB of Q and dO per head).
constexpr long long kBwdHeadGroupBytes = 32ll << 20;
__device__ __forceinline__ int bwd_unit(int unit, int n_t, int bh_count, int hg, int* bh) {
  const int group = unit / (hg * n_t);
  const int within = unit - group * hg * n_t;
  const int here = min(hg, bh_count - group * hg);
  *bh = group * hg + within % here;
  return within / here;
}

// Visible keys of sequence b (key padding), all keys otherwise.
__device__ __forceinline__ int kv_len_of(const BwdParams& p, int b) {
  int n = p.Lk;
  if (masks_padding(p.mask_kind)) {
    const int len = __ldg(p.key_lens + b);
    n = len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
  }
  return n;
}

// ---------------------------------------------------------------------------
// dK, dV: units (b, h, key tile), persistent CTAs
// ---------------------------------------------------------------------------
// The grid has one CTA per unit, but a running CTA cancels CTAs that have not
// started (cluster launch control) and takes their units, as the forward
// does: the TMA warp loads the next unit's K and V as soon as the current
// unit's last score products are done with them, and the next unit's first
// score products are issued while the gradient warps still write the current
// unit's dK and dV, so the per-CTA set-up, the K/V load latency and the
// pipeline fill leave the critical path.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int id) { return s_base + C::OFF_BAR + 8u * id; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  const uint32_t clc_resp = s_base + C::OFF_MISC + 16;
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);

  const int n_kt = (p.Lk + 127) / 128;
  const int n_qt = (p.Lq + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(bar(kFixFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kRingFull + s), 1);
      mbar_init(bar(kRingEmpty + s), 1);
      mbar_init(bar(kUnitFull + s), 1);
      mbar_init(bar(kUnitEmpty + s), kBwdUnitConsumers);
    }
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(bar(kScores + hf), 1);
      mbar_init(bar(kGrads + hf), kGradThreads);
    }
    mbar_init(bar(kAccDone), 1);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kFixFree), 1);
    mbar_init(bar(kAccFree), kGradThreads);
    mbar_init(bar(kClc), 1);
    mbar_init(bar(kStgFull), kGradThreads);
    mbar_init(bar(kStgFree), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // global memory only from here on (the set-up may overlap the previous
  // kernel on the stream, which for this kernel writes D)
  griddep_wait();

  // a unit's geometry: first key tile first (under the causal mask it sees
  // the most query tiles)
  struct KvUnit {
    int b, h, k0, qt_begin, n_iter, kv_len;
  };
  auto decode = [&](int unit) {
    KvUnit u;
    int bh = 0;
    const int kt = bwd_unit(unit, n_kt, p.B * p.H, p.head_group, &bh);
    u.b = bh / p.H;
    u.h = bh % p.H;
    u.k0 = kt * 128;
    u.kv_len = kv_len_of(p, u.b);
    // query tiles that see a key of this tile (causal: from the diagonal on)
    u.qt_begin = masks_causal(p.mask_kind) ? kt : 0;
    u.n_iter = (u.k0 < u.kv_len) ? (n_qt - u.qt_begin) : 0;
    return u;
  };
  // the k-th unit of this CTA from the queue (-1: no more, or gave up)
  auto take = [&](int k, int role) {
    const int slot = k & 1;
    if (!mbar_wait(bar(kUnitFull + slot), (k >> 1) & 1, abort_flag, p.status,
                   role * 64 + kUnitFull + slot))
      return -1;
    return static_cast<int>(unit_slot[slot]);
  };
  auto release = [&](int k) { mbar_arrive(bar(kUnitEmpty + (k & 1))); };

  if (warp == kSchedWarp) {
    // ---- scheduler (one lane): publishes the CTA's own unit, then keeps one
    // unit of look-ahead by cancelling CTAs that have not started
    if (lane == 0) {
      int unit = static_cast<int>(blockIdx.x);
      for (int k = 0;; ++k) {
        const int slot = k & 1;
        if (k >= 2 && !mbar_wait(bar(kUnitEmpty + slot), ((k >> 1) - 1) & 1, abort_flag, p.status,
                                 kRoleBwdSched * 64 + kUnitEmpty + slot))
          unit = -1;
        unit_slot[slot] = unit;
        mbar_arrive(bar(kUnitFull + slot));
        if (unit < 0) break;
        mbar_arrive_expect_tx(bar(kClc), 16);
        clc_try_cancel(clc_resp, bar(kClc));
        // the response is written asynchronously: wait for it even when the
        // CTA is giving up, so nothing lands in shared memory after exit
        volatile int never = 0;
        if (!mbar_wait(bar(kClc), k & 1, &never, p.status, kRoleBwdSched * 64 + kClc) ||
            *abort_flag)
          unit = -1;
        else
          unit = clc_query_first_ctaid_x(clc_resp);
      }
    }
    __syncwarp();
  } else if (warp == kTmaWarp) {
    // ---- TMA (one lane): per unit K and V (once the previous unit's last
    // score products are done with them), then Q_i, dO_i per query tile
    if (lane == 0) {
      int ring_t = 0;  // query tiles issued so far, over all units
      int fix_n = 0;   // units whose K and V were loaded
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int unit = take(k, kRoleBwdProducer);
        if (unit >= 0) release(k);
        if (unit < 0) break;
        const KvUnit u = decode(unit);
        if (u.n_iter == 0) continue;
        if (fix_n > 0 && !mbar_wait(bar(kFixFree), (fix_n - 1) & 1, abort_flag, p.status,
                                    kRoleBwdProducer * 64 + kFixFree))
          break;
        mbar_arrive_expect_tx(bar(kFixFull), 2 * C::TILE);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_4d(s_base + C::OFF_A0 + c * C::CHUNK, &p.tm_k, bar(kFixFull), 64 * c, u.h, u.k0, u.b);
          tma_load_4d(s_base + C::OFF_A1 + c * C::CHUNK, &p.tm_v, bar(kFixFull), 64 * c, u.h, u.k0, u.b);
        }
        ++fix_n;
        for (int it = 0; it < u.n_iter; ++it, ++ring_t) {
          const int s = ring_t & 1;
          if (ring_t >= 2 && !mbar_wait(bar(kRingEmpty + s), ((ring_t >> 1) - 1) & 1, abort_flag,
                                        p.status, kRoleBwdProducer * 64 + s)) {
            ok = false;
            break;
          }
          const int q0 = (u.qt_begin + it) * 128;
          const uint32_t dst = s_base + C::OFF_RING + s * 2 * C::TILE;
          mbar_arrive_expect_tx(bar(kRingFull + s), 2 * C::TILE);
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_4d(dst + c * C::CHUNK, &p.tm_q, bar(kRingFull + s), 64 * c, u.h, q0, u.b);
            tma_load_4d(dst + C::TILE + c * C::CHUNK, &p.tm_do, bar(kRingFull + s), 64 * c, u.h, q0,
                        u.b);
          }
        }
      }
      // every copy started lands before the CTA exits
      volatile int never = 0;
      if (fix_n > 0)
        mbar_wait(bar(kFixFull), (fix_n - 1) & 1, &never, p.status, kRoleBwdProducer * 64 + 8);
      for (int t = (ring_t > 2 ? ring_t - 2 : 0); t < ring_t; ++t)
        mbar_wait(bar(kRingFull + (t & 1)), (t >> 1) & 1, &never, p.status,
                  kRoleBwdProducer * 64 + 9);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer.  A query tile is taken in two halves of 64 queries with
    // score regions of their own, so the tensor cores work on one half while
    // the gradient warps work on the other: per half, dV/dK of this tile, then
    // S^T/dP^T of the next tile into the region just consumed.  Across units
    // the next unit's first score products follow the current unit's last
    // accumulating products the same way; only its first accumulating product
    // waits for the epilogue to have read dK and dV.
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);   // K-major A and B
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);     // B MN-major
    const uint64_t dA0 = smem_desc_sw128(s_base + C::OFF_A0, 16, 1024);   // K tile, K-major
    const uint64_t dA1 = smem_desc_sw128(s_base + C::OFF_A1, 16, 1024);   // V tile, K-major
    // queries 64 hf .. 64 hf + 63 of ring stage (t & 1): 64 rows of 128 bytes on
    auto half_rows = [&](int t, int hf) {
      return s_base + C::OFF_RING + (t & 1) * 2 * C::TILE + hf * 64 * 128;
    };
    // S^T = K Q^T, dP^T = V dO^T of half hf (keys on lanes, queries on columns)
    auto issue_scores = [&](int t, int hf) {
      const uint32_t rows = half_rows(t, hf);
      const uint64_t dQk = smem_desc_sw128(rows, 16, 1024);
      const uint64_t dDk = smem_desc_sw128(rows + C::TILE, 16, 1024);
      const uint32_t ts = tmem + C::TM_HALF * hf;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ss(ts, dA0 + off, dQk + off, idesc_s, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ss(ts + C::TM_DP, dA1 + off, dDk + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(bar(kScores + hf));
    };
    // dV += P^T dO, dK += dS^T Q over half hf.  The 16 queries of step ks are
    // 8 packed TMEM columns: chunk ks of the half (one gradient warp's 16
    // columns) keeps them in its first 8.
    auto issue_grads = [&](int t, int hf, bool first) {
      const uint32_t rows = half_rows(t, hf);
      const uint64_t dQm = smem_desc_sw128(rows, C::CHUNK, 1024);
      const uint64_t dDm = smem_desc_sw128(rows + C::TILE, C::CHUNK, 1024);
      const uint32_t ts = tmem + C::TM_HALF * hf;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ts(tmem + C::TM_ACC0, ts + a_col(ks), dDm + static_cast<uint64_t>((ks * 2048) >> 4),
                idesc_o, (ks > 0 || !first) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ts(tmem + C::TM_ACC1, ts + C::TM_DP + a_col(ks), dQm + static_cast<uint64_t>((ks * 2048) >> 4),
                idesc_o, (ks > 0 || !first) ? 1u : 0u);
    };
    bool ok = true;
    int ring_t = 0;  // query tiles of the units before the current one
    int fix_n = 0;   // units with work so far
    for (int k = 0; ok; ++k) {
      const int unit = take(k, kRoleBwdMma);
      __syncwarp();
      if (unit >= 0 && lane == 0) release(k);
      if (unit < 0) break;
      const KvUnit u = decode(unit);
      if (u.n_iter == 0) continue;
      ok = mbar_wait(bar(kFixFull), fix_n & 1, abort_flag, p.status, kRoleBwdMma * 64 + kFixFull) &&
           mbar_wait(bar(kRingFull + (ring_t & 1)), (ring_t >> 1) & 1, abort_flag, p.status,
                     kRoleBwdMma * 64 + kRingFull);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        issue_scores(ring_t, 0);
        issue_scores(ring_t, 1);
        // a one-tile unit's score products are its last use of K and V
        if (u.n_iter == 1) umma_commit(bar(kFixFree));
      }
      __syncwarp();
      for (int it = 0; ok && it < u.n_iter; ++it) {
        const int t = ring_t + it;
        const bool more = it + 1 < u.n_iter;
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(bar(kGrads + hf), t & 1, abort_flag, p.status,
                         kRoleBwdMma * 64 + kGrads + hf)) {
            ok = false;
            break;
          }
          // the unit's first accumulating product overwrites dK and dV: the
          // previous unit's epilogue must have read them
          if (it == 0 && hf == 0 && fix_n > 0 &&
              !mbar_wait(bar(kAccFree), (fix_n - 1) & 1, abort_flag, p.status,
                         kRoleBwdMma * 64 + kAccFree)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_grads(t, hf, it == 0 && hf == 0);
            if (hf == 1) {
              umma_commit(bar(kRingEmpty + (t & 1)));
              if (!more) umma_commit(bar(kAccDone));
            }
          }
          __syncwarp();
          if (!more) continue;
          const int sn = (t + 1) & 1;
          if (hf == 0 && !mbar_wait(bar(kRingFull + sn), ((t + 1) >> 1) & 1, abort_flag, p.status,
                                    kRoleBwdMma * 64 + kRingFull + sn)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_scores(t + 1, hf);
            // the last tile's score products are the unit's last use of K, V
            if (hf == 1 && it + 2 == u.n_iter) umma_commit(bar(kFixFree));
          }
          __syncwarp();
        }
      }
      ring_t += u.n_iter;
      ++fix_n;
    }
    if (elect_one()) umma_commit(bar(kDrain));
    __syncwarp();
    volatile int never = 0;
    mbar_wait(bar(kDrain), 0, &never, p.status, kRoleBwdMma * 64 + kDrain);
  } else {
    // ---- gradient warps: warp w owns key rows k0 + 32 (w % 4) .. (its TMEM
    // lane quarter) and, of each half tile, the 16 queries of chunk w / 4
    const int quarter = warp & 3, cq = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    // lse and D of the queries of this warp's chunk come straight from global
    // memory (every lane loads the same 64 bytes: one broadcast), as 16-byte
    // vectors when the rows are so aligned
    const bool vec_ok = p.Lq % 4 == 0 && (reinterpret_cast<uintptr_t>(p.lse) & 15u) == 0 &&
                        (reinterpret_cast<uintptr_t>(p.dvec) & 15u) == 0;
    bool ok = true;
    int ring_t = 0;  // query tiles of the units before the current one
    int unit_n = 0;  // units with work so far
    int stg_n = 0;   // epilogue chunks staged so far
    const uint32_t stg_v = s_base + C::OFF_STG, stg_k = stg_v + C::CHUNK;
    // The next unit is taken from the queue at the current unit's last tile.
    int next_unit_idx = -2;  // -2: not taken early
    for (int k = 0; ok; ++k) {
      int unit;
      if (next_unit_idx != -2) {
        unit = next_unit_idx;
        next_unit_idx = -2;
      } else {
        unit = take(k, kRoleBwdGrad);
        __syncwarp();
        if (unit >= 0 && lane == 0) release(k);
      }
      if (unit < 0) {
        ok = unit == -1 && !*abort_flag;
        break;
      }
      const KvUnit u = decode(unit);
      const int b = u.b, h = u.h, k0 = u.k0, qt_begin = u.qt_begin, n_iter = u.n_iter;
      const int kv_len = u.kv_len;
      const int key = k0 + r;
      const size_t vrow = (static_cast<size_t>(b) * p.H + h) * p.Lq;
      for (int it = 0; ok && it < n_iter; ++it) {
        const int t_all = ring_t + it;  // barrier phases run over all units
        const int q0 = (qt_begin + it) * 128;
        if (it + 1 == n_iter) {
          // last tile: the next unit now
          next_unit_idx = take(k + 1, kRoleBwdGrad);
          __syncwarp();
          if (next_unit_idx >= 0 && lane == 0) release(k + 1);
        }
        // Every (key, query) pair of the tile is visible unless the tile holds
        // keys past the key length, queries past Lq, or the causal diagonal.
        const bool all_visible = k0 + 127 < kv_len && q0 + 127 < p.Lq &&
                                 !(masks_causal(p.mask_kind) && q0 < k0 + 127);
        for (int hf = 0; hf < 2; ++hf) {
          const int col0 = 64 * hf + 16 * cq;  // first query column of the chunk
          const int qb = q0 + col0;
          // (loaded before the wait for the scores, so their latency is hidden)
          float l2c[16], dvc[16];  // negated: -lse (log2 units), -D
          if (vec_ok && qb + 16 <= p.Lq) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const float4 lv = __ldg(reinterpret_cast<const float4*>(p.lse + vrow + qb) + v4);
              const float4 dv = __ldg(reinterpret_cast<const float4*>(p.dvec + vrow + qb) + v4);
              l2c[4 * v4] = lv.x, l2c[4 * v4 + 1] = lv.y, l2c[4 * v4 + 2] = lv.z, l2c[4 * v4 + 3] = lv.w;
              dvc[4 * v4] = dv.x, dvc[4 * v4 + 1] = dv.y, dvc[4 * v4 + 2] = dv.z, dvc[4 * v4 + 3] = dv.w;
            }
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const bool in = qb + t < p.Lq;
              l2c[t] = in ? __ldg(p.lse + vrow + qb + t) : -INFINITY;
              dvc[t] = in ? __ldg(p.dvec + vrow + qb + t) : 0.f;
            }
          }
          if (!mbar_wait(bar(kScores + hf), t_all & 1, abort_flag, p.status,
                         kRoleBwdGrad * 64 + kScores + hf)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ts = tmem + C::TM_HALF * hf + lane_off + 16u * cq;
          uint32_t sr[16], pr[16];
          tmem_ld16(ts, sr);
          tmem_ld16(ts + C::TM_DP, pr);
          tmem_ld_wait();
          // the loads issued before the wait are consumed only now
#pragma unroll
          for (int t = 0; t < 16; t += 2) {
            mul2(l2c[t], l2c[t + 1], l2c[t], l2c[t + 1], -1.4426950408889634f, -1.4426950408889634f);
            dvc[t] = -dvc[t];
            dvc[t + 1] = -dvc[t + 1];
          }
          float pf[16];
          // (the mask test stays outside the element loops, which then have no
          // branches and interleave their 16 independent chains; packed f32x2
          // arithmetic halves the issue slots of the float math)
          if (all_visible) {
#pragma unroll
            for (int t = 0; t < 16; t += 2) {
              fma2(pf[t], pf[t + 1], __uint_as_float(sr[t]), __uint_as_float(sr[t + 1]), c2, c2,
                   l2c[t], l2c[t + 1]);
              pf[t] = ex2_approx(pf[t]);
              pf[t + 1] = ex2_approx(pf[t + 1]);
            }
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const int qi = q0 + col0 + t;
              const bool vis = key < kv_len && qi < p.Lq &&
                               !(masks_causal(p.mask_kind) && key > qi) && l2c[t] != INFINITY;
              const float e = ex2_approx(fmaf(__uint_as_float(sr[t]), c2, l2c[t]));
              pf[t] = vis ? e : 0.f;
            }
          }
          // P^T in bf16 for the dV product; dS = P (dP - D) from the float32 P
          uint32_t pk[8], dk[8];
#pragma unroll
          for (int t = 0; t < 16; t += 2) {
            pk[t >> 1] = pack_bf16x2(pf[t], pf[t + 1]);
            float g0, g1;
            add2(g0, g1, __uint_as_float(pr[t]), __uint_as_float(pr[t + 1]), dvc[t], dvc[t + 1]);
            mul2(g0, g1, pf[t], pf[t + 1], g0, g1);
            dk[t >> 1] = pack_bf16x2(g0, g1);
          }
          // P^T over the first 8 of the chunk's S^T columns, dS^T over the first
          // 8 of its dP^T columns (this thread has read them; no other has)
          tmem_st8(ts, pk);
          tmem_st8(ts + C::TM_DP, dk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(kGrads + hf));
        }
      }
      if (!ok) break;
      // ---- epilogue: dV and scale * dK rows to global (rows past Lk skipped);
      // warp w takes the 16-column chunks c with c % 4 == w / 4.  The
      // accumulators are read first, then released to the next unit.
      if (n_iter > 0) {
        ok = mbar_wait(bar(kAccDone), unit_n & 1, abort_flag, p.status,
                       kRoleBwdGrad * 64 + kAccDone);
        if (!ok) break;
        tc_fence_after();
      }
      // Per 64-column chunk: the accumulators to bf16 (dK scaled) in the
      // two staging buffers (128-byte swizzle, this thread's row and 32 of
      // the columns), then one thread stores both with TMA (rows past Lk and
      // columns past d are not written).  Row-wise global stores from each
      // thread cost this kernel about 9 % at d 128.
#pragma unroll 1
      for (int c64 = 0; c64 < C::KCH; ++c64) {
        const int c16 = 4 * c64 + cq;
        uint32_t a[16], kk[16];
        if (n_iter > 0) {
          tmem_ld16(tmem + C::TM_ACC0 + lane_off + 16u * c16, a);
          tmem_ld16(tmem + C::TM_ACC1 + lane_off + 16u * c16, kk);
          tmem_ld_wait();
          if (c64 + 1 == C::KCH) {
            // this thread's last accumulator columns are read: the next unit
            // may overwrite them
            tc_fence_before();
            mbar_arrive(bar(kAccFree));
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) a[t] = kk[t] = 0u;
        }
        // the previous chunk's stores must have read the staging buffers
        if (stg_n > 0 && !mbar_wait(bar(kStgFree), (stg_n - 1) & 1, abort_flag, p.status,
                                    kRoleBwdGrad * 64 + kStgFree)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int v4 = 0; v4 < 2; ++v4) {
          const uint32_t off = static_cast<uint32_t>(r * 128 + (((2 * cq + v4) ^ (r & 7)) << 4));
          st_shared_v4(stg_v + off,
                       pack_bf16x2(__uint_as_float(a[8 * v4 + 0]), __uint_as_float(a[8 * v4 + 1])),
                       pack_bf16x2(__uint_as_float(a[8 * v4 + 2]), __uint_as_float(a[8 * v4 + 3])),
                       pack_bf16x2(__uint_as_float(a[8 * v4 + 4]), __uint_as_float(a[8 * v4 + 5])),
                       pack_bf16x2(__uint_as_float(a[8 * v4 + 6]), __uint_as_float(a[8 * v4 + 7])));
          st_shared_v4(stg_k + off,
                       pack_bf16x2(__uint_as_float(kk[8 * v4 + 0]) * p.scale, __uint_as_float(kk[8 * v4 + 1]) * p.scale),
                       pack_bf16x2(__uint_as_float(kk[8 * v4 + 2]) * p.scale, __uint_as_float(kk[8 * v4 + 3]) * p.scale),
                       pack_bf16x2(__uint_as_float(kk[8 * v4 + 4]) * p.scale, __uint_as_float(kk[8 * v4 + 5]) * p.scale),
                       pack_bf16x2(__uint_as_float(kk[8 * v4 + 6]) * p.scale, __uint_as_float(kk[8 * v4 + 7]) * p.scale));
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kStgFull));
        if (threadIdx.x == 0) {
          if (!mbar_wait(bar(kStgFull), stg_n & 1, abort_flag, p.status,
                         kRoleBwdGrad * 64 + kStgFull)) {
            ok = false;
            break;
          }
          tma_store_4d(&p.tm_dv, stg_v, 64 * c64, h, k0, b);
          tma_store_4d(&p.tm_dk, stg_k, 64 * c64, h, k0, b);
          tma_store_commit();
          tma_store_wait_read();
          mbar_arrive(bar(kStgFree));
        }
        ++stg_n;
      }
      if (!ok) break;
      if (n_iter > 0) {
        ring_t += n_iter;
        ++unit_n;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// dQ: units (b, h, query tile), persistent CTAs
// ---------------------------------------------------------------------------
// Persistent like the dK/dV kernel: the TMA warp loads the next unit's Q and
// dO as soon as the current unit's last score products are done with them,
// and the next unit's first score products are issued while the gradient
// warps still write the current unit's dQ.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int id) { return s_base + C::OFF_BAR + 8u * id; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  const uint32_t clc_resp = s_base + C::OFF_MISC + 16;
  float* d_part = reinterpret_cast<float*>(smem + C::OFF_VEC);  // [2][128]
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);

  const int n_qt = (p.Lq + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(bar(kFixFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kRingFull + s), 1);
      mbar_init(bar(kRingEmpty + s), 1);
      mbar_init(bar(kUnitFull + s), 1);
      mbar_init(bar(kUnitEmpty + s), kBwdUnitConsumers);
    }
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(bar(kScores + hf), 1);
      mbar_init(bar(kGrads + hf), kGradThreads);
    }
    mbar_init(bar(kAccDone), 1);
    mbar_init(bar(kDrain), 1);
    mbar_init(bar(kAccFree), kGradThreads);
    mbar_init(bar(kClc), 1);
    mbar_init(bar(kOFree), kGradThreads);
    mbar_init(bar(kQTmem), kGradThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // global memory only from here on (the set-up may overlap the previous
  // kernel on the stream)
  griddep_wait();

  // a unit's geometry: last query tile first (under the causal mask it sees
  // the most key tiles)
  struct QUnit {
    int b, h, q0, qt, n_iter, kv_len;
  };
  auto decode = [&](int unit) {
    QUnit u;
    int bh = 0;
    u.qt = n_qt - 1 - bwd_unit(unit, n_qt, p.B * p.H, p.head_group, &bh);
    u.b = bh / p.H;
    u.h = bh % p.H;
    u.q0 = u.qt * 128;
    u.kv_len = kv_len_of(p, u.b);
    int n = (u.kv_len + 127) / 128;
    if (masks_causal(p.mask_kind) && n > u.qt + 1) n = u.qt + 1;
    u.n_iter = n;
    return u;
  };
  // the k-th unit of this CTA from the queue (-1: no more, or gave up)
  auto take = [&](int k, int role) {
    const int slot = k & 1;
    if (!mbar_wait(bar(kUnitFull + slot), (k >> 1) & 1, abort_flag, p.status,
                   role * 64 + kUnitFull + slot))
      return -1;
    return static_cast<int>(unit_slot[slot]);
  };
  auto release = [&](int k) { mbar_arrive(bar(kUnitEmpty + (k & 1))); };

  if (warp == kSchedWarp) {
    // ---- scheduler (one lane): publishes the CTA's own unit, then keeps one
    // unit of look-ahead by cancelling CTAs that have not started
    if (lane == 0) {
      int unit = static_cast<int>(blockIdx.x);
      for (int k = 0;; ++k) {
        const int slot = k & 1;
        if (k >= 2 && !mbar_wait(bar(kUnitEmpty + slot), ((k >> 1) - 1) & 1, abort_flag, p.status,
                                 kRoleBwdSched * 64 + kUnitEmpty + slot))
          unit = -1;
        unit_slot[slot] = unit;
        mbar_arrive(bar(kUnitFull + slot));
        if (unit < 0) break;
        mbar_arrive_expect_tx(bar(kClc), 16);
        clc_try_cancel(clc_resp, bar(kClc));
        // the response is written asynchronously: wait for it even when the
        // CTA is giving up, so nothing lands in shared memory after exit
        volatile int never = 0;
        if (!mbar_wait(bar(kClc), k & 1, &never, p.status, kRoleBwdSched * 64 + kClc) ||
            *abort_flag)
          unit = -1;
        else
          unit = clc_query_first_ctaid_x(clc_resp);
      }
    }
    __syncwarp();
  } else if (warp == kTmaWarp) {
    // ---- TMA (one lane): per unit Q and dO (once the previous unit's last
    // score products are done with them), then K_j, V_j per key tile
    if (lane == 0) {
      int ring_t = 0;  // key tiles issued so far, over all units
      int fix_n = 0;   // units whose Q and dO were loaded
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int unit = take(k, kRoleBwdProducer);
        if (unit >= 0) release(k);
        if (unit < 0) break;
        const QUnit u = decode(unit);
        if (u.n_iter == 0) continue;
        // the previous unit's staged Q, dO and O must have been read (D
        // formed, Q and dO copied into TMEM); the score products never read
        // them from shared memory
        if (fix_n > 0 && !mbar_wait(bar(kOFree), (fix_n - 1) & 1, abort_flag, p.status,
                                    kRoleBwdProducer * 64 + 16 + kOFree))
          break;
        mbar_arrive_expect_tx(bar(kFixFull), 3 * C::TILE);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_4d(s_base + C::OFF_A0 + c * C::CHUNK, &p.tm_q, bar(kFixFull), 64 * c, u.h, u.q0, u.b);
          tma_load_4d(s_base + C::OFF_A1 + c * C::CHUNK, &p.tm_do, bar(kFixFull), 64 * c, u.h, u.q0,
                      u.b);
          tma_load_4d(s_base + C::OFF_O + c * C::CHUNK, &p.tm_o, bar(kFixFull), 64 * c, u.h, u.q0, u.b);
        }
        ++fix_n;
        for (int it = 0; it < u.n_iter; ++it, ++ring_t) {
          const int s = ring_t & 1;
          if (ring_t >= 2 && !mbar_wait(bar(kRingEmpty + s), ((ring_t >> 1) - 1) & 1, abort_flag,
                                        p.status, kRoleBwdProducer * 64 + 16 + s)) {
            ok = false;
            break;
          }
          const int k0 = it * 128;
          const uint32_t dst = s_base + C::OFF_RING + s * 2 * C::TILE;
          mbar_arrive_expect_tx(bar(kRingFull + s), 2 * C::TILE);
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_4d(dst + c * C::CHUNK, &p.tm_k, bar(kRingFull + s), 64 * c, u.h, k0, u.b);
            tma_load_4d(dst + C::TILE + c * C::CHUNK, &p.tm_v, bar(kRingFull + s), 64 * c, u.h, k0,
                        u.b);
          }
        }
      }
      volatile int never = 0;
      if (fix_n > 0)
        mbar_wait(bar(kFixFull), (fix_n - 1) & 1, &never, p.status, kRoleBwdProducer * 64 + 24);
      for (int t = (ring_t > 2 ? ring_t - 2 : 0); t < ring_t; ++t)
        mbar_wait(bar(kRingFull + (t & 1)), (t >> 1) & 1, &never, p.status,
                  kRoleBwdProducer * 64 + 25);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer, in halves of 64 keys as in the dK/dV kernel
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
    // keys 64 hf .. 64 hf + 63 of ring stage (t & 1)
    auto half_rows = [&](int t, int hf) {
      return s_base + C::OFF_RING + (t & 1) * 2 * C::TILE + hf * 64 * 128;
    };
    // S = Q K^T, dP = dO V^T of half hf (queries on lanes, keys on columns)
    auto issue_scores = [&](int t, int hf) {
      const uint32_t rows = half_rows(t, hf);
      const uint64_t dKk = smem_desc_sw128(rows, 16, 1024);
      const uint64_t dVk = smem_desc_sw128(rows + C::TILE, 16, 1024);
      const uint32_t ts = tmem + C::TM_HALF * hf;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ts(ts, tmem + C::TM_QA + 8u * ks, dKk + off, idesc_s, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = static_cast<uint64_t>((((ks >> 2) * C::CHUNK) + (ks & 3) * 32) >> 4);
        umma_ts(ts + C::TM_DP, tmem + C::TM_DOA + 8u * ks, dVk + off, idesc_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(bar(kScores + hf));
    };
    // dQ += dS K over half hf (16 keys = 8 packed TMEM columns of A per step)
    auto issue_grads = [&](int t, int hf, bool first) {
      const uint64_t dKm = smem_desc_sw128(half_rows(t, hf), C::CHUNK, 1024);  // K, MN-major
      const uint32_t ts = tmem + C::TM_HALF * hf;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_ts(tmem + C::TM_ACC0, ts + a_col(ks), dKm + static_cast<uint64_t>((ks * 2048) >> 4),
                idesc_o, (ks > 0 || !first) ? 1u : 0u);
    };
    bool ok = true;
    int ring_t = 0;  // key tiles of the units before the current one
    int fix_n = 0;   // units with work so far
    for (int k = 0; ok; ++k) {
      const int unit = take(k, kRoleBwdMma);
      __syncwarp();
      if (unit >= 0 && lane == 0) release(k);
      if (unit < 0) break;
      const QUnit u = decode(unit);
      if (u.n_iter == 0) continue;
      // the unit's Q and dO in TMEM (the gradient warps copy them)
      ok = mbar_wait(bar(kQTmem), fix_n & 1, abort_flag, p.status,
                     kRoleBwdMma * 64 + 16 + kQTmem) &&
           mbar_wait(bar(kRingFull + (ring_t & 1)), (ring_t >> 1) & 1, abort_flag, p.status,
                     kRoleBwdMma * 64 + 16 + kRingFull);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        issue_scores(ring_t, 0);
        issue_scores(ring_t, 1);
      }
      __syncwarp();
      for (int it = 0; ok && it < u.n_iter; ++it) {
        const int t = ring_t + it;
        const bool more = it + 1 < u.n_iter;
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(bar(kGrads + hf), t & 1, abort_flag, p.status,
                         kRoleBwdMma * 64 + 16 + kGrads + hf)) {
            ok = false;
            break;
          }
          // the unit's first accumulating product overwrites dQ: the previous
          // unit's epilogue must have read it
          if (it == 0 && hf == 0 && fix_n > 0 &&
              !mbar_wait(bar(kAccFree), (fix_n - 1) & 1, abort_flag, p.status,
                         kRoleBwdMma * 64 + 16 + kAccFree)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_grads(t, hf, it == 0 && hf == 0);
            if (hf == 1) {
              umma_commit(bar(kRingEmpty + (t & 1)));
              if (!more) umma_commit(bar(kAccDone));
            }
          }
          __syncwarp();
          if (!more) continue;
          const int sn = (t + 1) & 1;
          if (hf == 0 && !mbar_wait(bar(kRingFull + sn), ((t + 1) >> 1) & 1, abort_flag, p.status,
                                    kRoleBwdMma * 64 + 16 + kRingFull + sn)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) issue_scores(t + 1, hf);
          __syncwarp();
        }
      }
      ring_t += u.n_iter;
      ++fix_n;
    }
    if (elect_one()) umma_commit(bar(kDrain));
    __syncwarp();
    volatile int never = 0;
    mbar_wait(bar(kDrain), 0, &never, p.status, kRoleBwdMma * 64 + 16 + kDrain);
  } else {
    // ---- gradient warps: warp w owns query rows q0 + 32 (w % 4) .. and, of
    // each half tile, the 16 keys of chunk w / 4
    const int quarter = warp & 3, cq = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    bool ok = true;
    int ring_t = 0;  // key tiles of the units before the current one
    int unit_n = 0;  // units with work whose epilogue ran
    int prep_n = 0;  // units with work prepared
    // dQ rows in whole 32-byte sectors: rows of a multiple of 16 elements
    // from a 32-byte aligned base
    const bool whole_sectors =
        p.d % 16 == 0 && (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0;
    // Prepares a unit with key tiles once its Q, dO and O are staged: D_i =
    // dO_i . O_i of this row (the warps of chunks 0 and 1 of the lane quarter
    // take alternate 16-byte pieces and add their halves in shared memory; it
    // is also written to the workspace for the dK/dV kernel, which runs next),
    // the row's lse, and this warp's 32 columns of the unit's Q (chunks 0, 1)
    // or dO (2, 3) copied into TMEM, where the score products read them.  The
    // staged tiles are then free for the following unit's.
    auto prepare = [&](const QUnit& w, float* l2_out, float* dvv_out) -> bool {
      const int qi = w.q0 + r;
      const size_t idx = (static_cast<size_t>(w.b) * p.H + w.h) * p.Lq + qi;
      float l2 = -INFINITY, part = 0.f;
      if (qi < p.Lq) l2 = p.lse[idx] * 1.4426950408889634f;
      if (!mbar_wait(bar(kFixFull), prep_n & 1, abort_flag, p.status,
                     kRoleBwdGrad * 64 + 16 + kFixFull))
        return false;
      const int pieces = p.d / 8;  // the tiles hold zeros past d
      for (int c = cq; cq < 2 && c < pieces; c += 2) {
        const uint32_t off = static_cast<uint32_t>((c >> 3) * C::CHUNK + r * 128 +
                                                   (((c & 7) ^ (r & 7)) << 4));
        const uint4 ov = ld_shared_v4(s_base + C::OFF_O + off);
        const uint4 gv = ld_shared_v4(s_base + C::OFF_A1 + off);
        part += bf_lo(ov.x) * bf_lo(gv.x) + bf_hi(ov.x) * bf_hi(gv.x) + bf_lo(ov.y) * bf_lo(gv.y) +
                bf_hi(ov.y) * bf_hi(gv.y) + bf_lo(ov.z) * bf_lo(gv.z) + bf_hi(ov.z) * bf_hi(gv.z) +
                bf_lo(ov.w) * bf_lo(gv.w) + bf_hi(ov.w) * bf_hi(gv.w);
      }
      // (the previous unit's score products, the last readers of these TMEM
      // columns, are complete: this warp waited for every one of them)
      const int c = cq & 1;
      if (c < C::KCH) {
        const uint32_t src = s_base + (cq < 2 ? C::OFF_A0 : C::OFF_A1) + c * C::CHUNK + r * 128;
        uint32_t wd[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = ld_shared_v4(src + (static_cast<uint32_t>(v ^ (r & 7)) << 4));
          wd[4 * v] = x.x;
          wd[4 * v + 1] = x.y;
          wd[4 * v + 2] = x.z;
          wd[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + (cq < 2 ? C::TM_QA : C::TM_DOA) + 32u * c, wd);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(kQTmem));
      mbar_arrive(bar(kOFree));
      ++prep_n;
      if (cq < 2) d_part[cq * 128 + r] = part;
      // (the second barrier keeps the next unit's halves from overwriting
      // this one's before both warps of the quarter have read them.  A named
      // barrier cannot time out: after each one the abort flag is checked,
      // and a warp that gives up arrives once on it on its way out.)
      named_barrier(1, kGradThreads);
      if (*abort_flag) return false;
      const float dvv = d_part[r] + d_part[128 + r];
      named_barrier(1, kGradThreads);
      if (*abort_flag) return false;
      if (cq == 0 && qi < p.Lq) p.dvec[idx] = dvv;
      *l2_out = l2;
      *dvv_out = dvv;
      return true;
    };
    int unit = take(0, kRoleBwdGrad);
    __syncwarp();
    if (unit >= 0 && lane == 0) release(0);
    QUnit u{};
    float l2 = -INFINITY, dvv = 0.f;
    if (unit >= 0) {
      u = decode(unit);
      if (u.n_iter > 0) ok = prepare(u, &l2, &dvv);
    }
    if (unit == -1 && *abort_flag) ok = false;
    for (int k = 0; ok && unit >= 0; ++k) {
      const int b = u.b, h = u.h, q0 = u.q0, n_iter = u.n_iter, kv_len = u.kv_len;
      const int qi = q0 + r;
      const bool row_ok = qi < p.Lq && l2 != -INFINITY;
      for (int it = 0; ok && it < n_iter; ++it) {
        const int t_all = ring_t + it;  // barrier phases run over all units
        const int k0 = it * 128;
        // every key of the tile visible to every query of the unit's tile?
        const bool all_visible = k0 + 127 < kv_len && q0 + 127 < p.Lq &&
                                 !(masks_causal(p.mask_kind) && q0 < k0 + 127);
        for (int hf = 0; hf < 2; ++hf) {
          if (!mbar_wait(bar(kScores + hf), t_all & 1, abort_flag, p.status,
                         kRoleBwdGrad * 64 + 16 + kScores + hf)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ts = tmem + C::TM_HALF * hf + lane_off + 16u * cq;
          uint32_t sr[16], pr[16];
          tmem_ld16(ts, sr);
          tmem_ld16(ts + C::TM_DP, pr);
          tmem_ld_wait();
          float pf[16];
          if (all_visible) {
#pragma unroll
            for (int t = 0; t < 16; t += 2) {
              fma2(pf[t], pf[t + 1], __uint_as_float(sr[t]), __uint_as_float(sr[t + 1]), c2, c2,
                   -l2, -l2);
              pf[t] = ex2_approx(pf[t]);
              pf[t + 1] = ex2_approx(pf[t + 1]);
            }
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const int key = k0 + 64 * hf + 16 * cq + t;
              const bool vis = row_ok && key < kv_len && !(masks_causal(p.mask_kind) && key > qi);
              const float e = ex2_approx(fmaf(__uint_as_float(sr[t]), c2, -l2));
              pf[t] = vis ? e : 0.f;
            }
          }
          // dS = P (dP - D) from the float32 P (no product here takes P itself)
          uint32_t dk[8];
#pragma unroll
          for (int t = 0; t < 16; t += 2) {
            float g0, g1;
            add2(g0, g1, __uint_as_float(pr[t]), __uint_as_float(pr[t + 1]), -dvv, -dvv);
            mul2(g0, g1, pf[t], pf[t + 1], g0, g1);
            dk[t >> 1] = pack_bf16x2(g0, g1);
          }
          // dS over the first 8 of the chunk's S columns (read by this thread only)
          tmem_st8(ts, dk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(kGrads + hf));
        }
      }
      if (!ok) break;
      // The next unit is prepared before this unit's epilogue, so the tensor
      // cores start its first scores while the epilogue runs.
      const int unit_next = take(k + 1, kRoleBwdGrad);
      __syncwarp();
      if (unit_next >= 0 && lane == 0) release(k + 1);
      QUnit u_next{};
      float l2_next = -INFINITY, dvv_next = 0.f;
      if (unit_next >= 0) {
        u_next = decode(unit_next);
        if (u_next.n_iter > 0 && !prepare(u_next, &l2_next, &dvv_next)) {
          ok = false;
          break;
        }
      } else if (*abort_flag) {
        ok = false;
        break;
      }
      // ---- epilogue: the accumulator is read first, then released to the
      // next unit
      if (n_iter > 0) {
        ok = mbar_wait(bar(kAccDone), unit_n & 1, abort_flag, p.status,
                       kRoleBwdGrad * 64 + 16 + kAccDone);
        if (!ok) break;
        tc_fence_after();
      }
      __nv_bfloat16* dq_row = reinterpret_cast<__nv_bfloat16*>(p.dq) +
                              ((static_cast<size_t>(b) * p.Lq + qi) * p.H + h) * p.d;
#pragma unroll 1
      for (int c16 = cq; c16 < D / 16; c16 += 4) {
        uint32_t a[16];
        if (n_iter > 0) {
          tmem_ld16(tmem + C::TM_ACC0 + lane_off + 16u * c16, a);
          tmem_ld_wait();
          if (c16 + 4 >= D / 16) {
            // this thread's last accumulator columns are read
            tc_fence_before();
            mbar_arrive(bar(kAccFree));
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) a[t] = 0u;
        }
        if (qi < p.Lq) {
          uint4 w[2];
#pragma unroll
          for (int v4 = 0; v4 < 2; ++v4) {
            w[v4].x = pack_bf16x2(__uint_as_float(a[8 * v4 + 0]) * p.scale, __uint_as_float(a[8 * v4 + 1]) * p.scale);
            w[v4].y = pack_bf16x2(__uint_as_float(a[8 * v4 + 2]) * p.scale, __uint_as_float(a[8 * v4 + 3]) * p.scale);
            w[v4].z = pack_bf16x2(__uint_as_float(a[8 * v4 + 4]) * p.scale, __uint_as_float(a[8 * v4 + 5]) * p.scale);
            w[v4].w = pack_bf16x2(__uint_as_float(a[8 * v4 + 6]) * p.scale, __uint_as_float(a[8 * v4 + 7]) * p.scale);
          }
          if (whole_sectors && 16 * c16 + 16 <= p.d) {
            // one whole 32-byte sector
            st_global_v8(dq_row + 16 * c16, w[0], w[1]);
          } else {
#pragma unroll
            for (int v4 = 0; v4 < 2; ++v4) {
              if (16 * c16 + 8 * v4 >= p.d) break;  // columns past d are padding
              *reinterpret_cast<uint4*>(dq_row + 16 * c16 + 8 * v4) = w[v4];
            }
          }
        }
      }
      if (n_iter > 0) {
        ring_t += n_iter;
        ++unit_n;
      }
      unit = unit_next;
      u = u_next;
      l2 = l2_next;
      dvv = dvv_next;
    }
    if (!ok) named_barrier_arrive(1, kGradThreads);  // release gradient warps blocked on the barrier
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, cudaStream_t stream, LaunchInfo* info) {
  using C = BwdCfg<D>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_DKDV);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_DQ);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long bh = static_cast<long long>(p.B) * p.H;
  const long long kv_units = bh * ((p.Lk + 127) / 128);
  const long long q_units = bh * ((p.Lq + 127) / 128);
  // the dQ kernel forms D = dO . O for its rows and stores it; the dK/dV
  // kernel, next on the stream, reads it
  e = launch_serialized(bwd_dq_kernel<D>, dim3(static_cast<unsigned>(q_units)), dim3(kBwdThreads),
                        C::SMEM_DQ, stream, p);
  if (e != cudaSuccess) return e;
  e = launch_serialized(bwd_dkdv_kernel<D>, dim3(static_cast<unsigned>(kv_units)),
                        dim3(kBwdThreads), C::SMEM_DKDV, stream, p);
  if (info) {
    info->kernels = 2;
    info->grid = static_cast<int>(kv_units + q_units);
    info->block = kBwdThreads;
    info->smem = C::SMEM_DKDV > C::SMEM_DQ ? C::SMEM_DKDV : C::SMEM_DQ;
  }
  return e;
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& params, int d, cudaStream_t stream, LaunchInfo* info) {
  BwdParams p = params;
  {
    // bytes of the two tiles a head streams (Q and dO, or K and V)
    const long long L = p.Lq > p.Lk ? p.Lq : p.Lk;
    const long long per_head = 2ll * L * d * 2 > 0 ? 2ll * L * d * 2 : 1;
    long long hg = kBwdHeadGroupBytes / per_head;
    const long long bh = static_cast<long long>(p.B) * p.H;
    if (hg > bh) hg = bh;
    if (hg < 1) hg = 1;
    p.head_group = static_cast<int>(hg);
  }
  if (d == 64) return launch_bwd_d<64>(p, stream, info);
  if (d == 128) return launch_bwd_d<128>(p, stream, info);
  return cudaErrorInvalidValue;
}

}  // namespace mha
