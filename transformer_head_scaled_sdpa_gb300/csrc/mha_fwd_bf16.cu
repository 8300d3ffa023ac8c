// mha_fwd_bf16.cu -- bf16 attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Computes, for every (sequence b, head h, 128-query tile), the tile of
//   O = softmax(Q K^T * scale) V
// ("Attention Is All You Need", Section 3.2.1, Equation (1); all heads in
// parallel, Section 3.2.2) without ever writing the score matrix to memory:
// K/V are streamed in 128-key tiles and the softmax is evaluated online, so
// for each query row the running maximum m and running sum l are carried
// across tiles and the partial output is rescaled by 2^(m_old - m_new) when
// the maximum grows.  Subtracting a running maximum is exact because adding
// one constant to all scores of a row leaves the weights unchanged (formula
// page transformer-attention, section 証明, weight-ratio step).  The scale is
// folded into the exponent base: p = 2^(s * scale * log2(e) - m).
//
// One CTA = one work unit (b, h, q-tile).  256 threads in four roles:
//   warp 0       TMA producer: Q once, then K_j/V_j into an NS-stage ring
//   warp 1       TMEM allocator and MMA issuer (one thread):
//                  S_j = Q K_j^T  -> TMEM (two 128-column buffers)
//                  O  += P_j V_j  -> TMEM (d columns)
//   warps 2-3    idle
//   warps 4-7    softmax: thread r owns query row r (TMEM lane r): reads S_j,
//                masks, updates m and l, rescales O, writes P_j (bf16) to
//                shared memory; finally the 1/l epilogue stores O.
// Masks: causal tiles above the diagonal are never loaded or computed; the
// diagonal tile and a ragged last key tile are masked per element (score set
// to -inf, so its weight is exactly 0: formula page, 応用, 先を読まない仕掛け).
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

template <int D>
struct Cfg {
  static constexpr int KCH = D / 64;             // 128-byte chunks along d
  static constexpr int CHUNK = 128 * 128;        // one [128 rows x 128 B] swizzled chunk
  static constexpr int TILE = KCH * CHUNK;       // one 128-row Q, K or V tile
  static constexpr int NS = (D == 64) ? 3 : 2;   // K/V ring stages
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_P = OFF_V + NS * TILE;
  static constexpr int OFF_BAR = OFF_P + 2 * CHUNK;  // P: 128 x 128 bf16
  static constexpr int NBAR = 6 + 2 * NS;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  // TMEM columns
  static constexpr uint32_t TM_S = 0;    // S buffers at 0 and 128
  static constexpr uint32_t TM_O = 256;  // O: D columns
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// barrier ids inside the barrier block
template <int NS>
struct Bars {
  static constexpr int Q = 0;
  static constexpr int KV_FULL = 1;           // + stage
  static constexpr int KV_EMPTY = 1 + NS;     // + stage
  static constexpr int S_FULL = 1 + 2 * NS;   // + buffer (2)
  static constexpr int P_FULL = 3 + 2 * NS;
  static constexpr int PV_DONE = 4 + 2 * NS;
  static constexpr int DRAIN = 5 + 2 * NS;
};

// role ids for the status "site" field
constexpr int kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3;

template <int D>
__global__ void __launch_bounds__(256, 1) fwd_bf16_kernel(const __grid_constant__ Bf16Params p) {
  using C = Cfg<D>;
  using BA = Bars<C::NS>;
  constexpr int NS = C::NS;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::OFF_Q;
  const uint32_t sK = s_base + C::OFF_K;
  const uint32_t sV = s_base + C::OFF_V;
  const uint32_t sP = s_base + C::OFF_P;
  const uint32_t s_bar = s_base + C::OFF_BAR;
  auto bar = [&](int id) -> uint32_t { return s_bar + 8u * static_cast<uint32_t>(id); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);

  // ---- work unit: heavy causal tiles are dispatched first ----------------
  const int bh_count = p.B * p.H;
  const int qt_idx = static_cast<int>(blockIdx.x) / bh_count;
  const int bh = static_cast<int>(blockIdx.x) % bh_count;
  const int q_tile = (p.mask_kind == kMaskCausal) ? (p.n_qtiles - 1 - qt_idx) : qt_idx;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int q0 = q_tile * kBlockM;
  int kv_len = p.Lk;
  if (p.mask_kind == kMaskKeyPadding) {
    const int len = __ldg(p.key_lens + b);
    kv_len = len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
  }
  int n_tiles = (kv_len + kBlockN - 1) / kBlockN;
  if (p.mask_kind == kMaskCausal && n_tiles > q_tile + 1) n_tiles = q_tile + 1;

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    mbar_init(bar(BA::Q), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(BA::KV_FULL + s), 1);
      mbar_init(bar(BA::KV_EMPTY + s), 1);
    }
    mbar_init(bar(BA::S_FULL + 0), 1);
    mbar_init(bar(BA::S_FULL + 1), 1);
    mbar_init(bar(BA::P_FULL), 128);
    mbar_init(bar(BA::PV_DONE), 1);
    mbar_init(bar(BA::DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // =================== TMA producer ===================
    if (lane == 0 && n_tiles > 0) {
      int issued[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) issued[s] = 0;
      mbar_arrive_expect_tx(bar(BA::Q), C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_load_4d(sQ + c * C::CHUNK, &p.tm_q, bar(BA::Q), 64 * c, h, q0, b);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % NS;
        if (j >= NS) {
          if (!mbar_wait(bar(BA::KV_EMPTY + s), ((j / NS) - 1) & 1, abort_flag, p.status,
                         kRoleProducer * 16 + BA::KV_EMPTY + s))
            break;
        }
        mbar_arrive_expect_tx(bar(BA::KV_FULL + s), 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(sK + s * C::TILE + c * C::CHUNK, &p.tm_k, bar(BA::KV_FULL + s), 64 * c, h,
                      j * kBlockN, b);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_4d(sV + s * C::TILE + c * C::CHUNK, &p.tm_v, bar(BA::KV_FULL + s), 64 * c, h,
                      j * kBlockN, b);
        ++issued[s];
      }
      // Leave only when every copy this thread started has landed (the
      // normal path finds them complete already).
      mbar_wait(bar(BA::Q), 0, abort_flag, p.status, kRoleProducer * 16 + BA::Q);
#pragma unroll
      for (int s = 0; s < NS; ++s)
        if (issued[s] > 0)
          mbar_wait(bar(BA::KV_FULL + s), (issued[s] - 1) & 1, abort_flag, p.status,
                    kRoleProducer * 16 + BA::KV_FULL + s);
    }
  } else if (warp == 1) {
    // =================== MMA issuer ===================
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      auto issue_s = [&](int j) {
        const int s = j % NS;
        const uint32_t d_tmem = tmem + C::TM_S + 128u * static_cast<uint32_t>(j & 1);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::CHUNK + (ks & 3) * 32;
          const uint64_t a = smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sK + s * C::TILE + off, 16, 1024);
          umma_ss(d_tmem, a, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int j) {
        const int s = j % NS;
#pragma unroll
        for (int ks = 0; ks < kBlockN / 16; ++ks) {
          const uint64_t a = smem_desc_sw128(sP + (ks >> 2) * C::CHUNK + (ks & 3) * 32, 16, 1024);
          // V is MN-major (d contiguous): 16 keys = 16 rows of 128 B; the
          // second 64-wide d chunk sits one CHUNK further.
          const uint64_t bd = smem_desc_sw128(sV + s * C::TILE + ks * 2048, C::CHUNK, 1024);
          umma_ss(tmem + C::TM_O, a, bd, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(BA::Q), 0, abort_flag, p.status, kRoleMma * 16 + BA::Q) &&
                mbar_wait(bar(BA::KV_FULL), 0, abort_flag, p.status, kRoleMma * 16 + BA::KV_FULL);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        umma_commit(bar(BA::S_FULL + 0));
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          const int s1 = (j + 1) % NS;
          ok = mbar_wait(bar(BA::KV_FULL + s1), ((j + 1) / NS) & 1, abort_flag, p.status,
                         kRoleMma * 16 + BA::KV_FULL + s1);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
          umma_commit(bar(BA::S_FULL + ((j + 1) & 1)));
        }
        ok = mbar_wait(bar(BA::P_FULL), j & 1, abort_flag, p.status, kRoleMma * 16 + BA::P_FULL);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j);
        umma_commit(bar(BA::PV_DONE));
        umma_commit(bar(BA::KV_EMPTY + (j % NS)));
      }
      // Every MMA this thread issued completes before TMEM is released.
      umma_commit(bar(BA::DRAIN));
      volatile int never = 0;
      mbar_wait(bar(BA::DRAIN), 0, &never, p.status, kRoleMma * 16 + BA::DRAIN);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // =================== softmax + epilogue ===================
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;          // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    const int qi = q0 + row;
    float m = -INFINITY;  // running max of s * scale * log2(e)
    float l = 0.f;        // running sum of 2^(s*c2 - m)
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int buf = j & 1;
      ok = mbar_wait(bar(BA::S_FULL + buf), (j >> 1) & 1, abort_flag, p.status,
                     kRoleSoftmax * 16 + BA::S_FULL + buf);
      if (!ok) break;
      tc_fence_after();
      uint32_t r[128];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        tmem_ld32(tmem + lane_off + C::TM_S + 128u * buf + 32u * c4,
                  *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c4]));
      tmem_ld_wait();
      float x[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(r[c]);
      // per-element mask on the diagonal tile and a ragged last tile
      const int kbase = j * kBlockN;
      int lim = kv_len - kbase;                                   // keys c < lim exist
      if (p.mask_kind == kMaskCausal && qi - kbase + 1 < lim) lim = qi - kbase + 1;
      if (lim < kBlockN) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) x[c] = -INFINITY;
      }
      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int c = 4; c < 128; c += 4) {
        mx0 = fmaxf(mx0, x[c]);
        mx1 = fmaxf(mx1, x[c + 1]);
        mx2 = fmaxf(mx2, x[c + 2]);
        mx3 = fmaxf(mx3, x[c + 3]);
      }
      const float m_new = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_use);
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        x[c] = ex2_approx(fmaf(x[c], c2, -m_use));
        x[c + 1] = ex2_approx(fmaf(x[c + 1], c2, -m_use));
        x[c + 2] = ex2_approx(fmaf(x[c + 2], c2, -m_use));
        x[c + 3] = ex2_approx(fmaf(x[c + 3], c2, -m_use));
        s0 += x[c];
        s1 += x[c + 1];
        s2 += x[c + 2];
        s3 += x[c + 3];
      }
      l = l * alpha + ((s0 + s1) + (s2 + s3));
      m = m_new;
      if (j > 0) {
        // PV_{j-1} must be complete before O is rescaled and P overwritten.
        ok = mbar_wait(bar(BA::PV_DONE), (j - 1) & 1, abort_flag, p.status,
                       kRoleSoftmax * 16 + BA::PV_DONE);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c32 = 0; c32 < D / 32; ++c32) {
            uint32_t o[32];
            const uint32_t addr = tmem + lane_off + C::TM_O + 32u * c32;
            tmem_ld32(addr, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(addr, o);
          }
          tmem_st_wait();
        }
      }
      // P_j as bf16, K-major with the 128-byte swizzle: keys 64c..64c+63 of
      // row `row` fill 128 bytes of chunk c; 16-byte unit u lands at u ^ (row % 8).
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t addr = sP + (u >> 3) * C::CHUNK + row * 128 +
                              ((static_cast<uint32_t>(u & 7) ^ (row & 7)) << 4);
        st_shared_v4(addr, pack_bf16x2(x[8 * u], x[8 * u + 1]),
                     pack_bf16x2(x[8 * u + 2], x[8 * u + 3]),
                     pack_bf16x2(x[8 * u + 4], x[8 * u + 5]),
                     pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(BA::P_FULL));
    }
    if (ok && n_tiles > 0) {
      ok = mbar_wait(bar(BA::PV_DONE), (n_tiles - 1) & 1, abort_flag, p.status,
                     kRoleSoftmax * 16 + BA::PV_DONE);
      tc_fence_after();
    }
    if (ok) {
      // epilogue: O / l rounded to bf16; rows past Lq are not stored
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<__nv_bfloat16*>(p.out) +
          ((static_cast<size_t>(b) * p.Lq + qi) * p.H + h) * D);
#pragma unroll
      for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_off + C::TM_O + 32u * c32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        if (qi < p.Lq) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[c32 * 4 + v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
        }
      }
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const Bf16Params& p, cudaStream_t stream, LaunchInfo* info) {
  using C = Cfg<D>;
  static bool attr_set = false;  // per process; the attribute is per function
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long units = static_cast<long long>(p.n_qtiles) * p.B * p.H;
  const dim3 grid(static_cast<unsigned>(units));
  fwd_bf16_kernel<D><<<grid, 256, C::SMEM, stream>>>(p);
  if (info) {
    info->kernels = 1;
    info->grid = static_cast<int>(units);
    info->block = 256;
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
