// mha_decode.cu -- attention for one new query per sequence over a key/value
// cache (decode step), bf16, sm_103a.
//
// At inference the decoder produces one token per step: the target sequence
// starts as <BOS>, each step appends the token it generated and runs the
// decoder again, and beam search keeps the best four sequences going
// (cookipedia article, section "Transformer 全体").  In the decoder's masked
// self-attention the usable length grows by one per step (D2L notes, the
// three kinds of attention, decoder layer A).  So a step's attention is, for
// each sequence b (one per beam) and head h, the single query row q of the
// new position against the n_b cached keys and values of positions
// 0 .. n_b - 1:
//   s_j = scale * (q . k_j),  o = sum_j softmax(s)_j v_j
// ("Attention Is All You Need", Section 3.2.1, Equation (1)) -- the forward
// with Lq = 1 and key lengths n_b.
//
// The work is reading the cache: 4 d_k bytes per key for 4 d_k flops, far
// below the tensor cores' balance point, so the kernel streams K and V from
// HBM with TMA and computes on the CUDA cores.  Keys are split into chunks
// processed by separate CTAs (split-K), so a small batch still has enough
// CTAs to keep every SM's loads in flight:
//   decode_split_kernel   grid (B*H, S): CTA (b*h, s) takes keys
//                         [s*C, min((s+1)*C, n_b)); four compute warps and a
//                         TMA warp stream 64-key tiles through a ring.  Each
//                         compute warp owns 16 keys of a tile and keeps its own
//                         running maximum m, sum l and unnormalised output; the
//                         four are merged at the end.  With S = 1 the CTA
//                         writes the output directly; otherwise it writes
//                         (o, m, l) to the workspace.
//   decode_combine_kernel one warp per (b, h): merges the S partial results
//                         exactly, o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
//                         with M = max_s m_s (adding a constant to all scores of
//                         a row changes no weight: formula page
//                         transformer-attention, section 証明).
// Scores are kept in log2 units (q is pre-multiplied by scale * log2(e)).
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

constexpr int kDecWarps = 4;                    // compute warps
constexpr int kDecThreads = 32 * (kDecWarps + 1);  // + the TMA warp
constexpr int kDecTile = 64;                    // keys per TMA tile
constexpr int kKeysPerWarp = kDecTile / kDecWarps;  // 16

// D: the kernel's width (64, 128 or 256); a head of d_k < D features runs on
// it with the rest of each row read as zero (the tensor maps' fill) and
// only its own d_k output columns written.
template <int D>
struct DecCfg {
  static constexpr int KCH = D / 64;              // 128-byte chunks per key row
  static constexpr int CHUNK = kDecTile * 128;    // [64 keys x 128 B], 128-byte swizzle
  static constexpr int TILE = KCH * CHUNK;        // one K or V tile
  static constexpr int NS = (D == 64) ? 4 : 3;    // ring stages (192 KB at D = 256)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = NS * TILE;
  static constexpr int OFF_BAR = 2 * NS * TILE;   // full[NS], empty[NS]
  static constexpr int OFF_ABORT = OFF_BAR + 16 * NS;
  static constexpr int OFF_RED = OFF_ABORT + 16;  // merge: m[4], l[4], o[4][D]
  static constexpr int SMEM = OFF_RED + (8 + kDecWarps * D) * 4 + 1024;
  static constexpr int EPL = D / 32;              // output elements per lane
  static_assert(OFF_V % 1024 == 0 && OFF_BAR % 8 == 0 && OFF_RED % 16 == 0, "alignment");
};

constexpr int kRoleDecProducer = 6, kRoleDecConsumer = 7;

// bf16 pairs -> float
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// This lane's EPL consecutive elements (from element EPL*lane) of key row r
// of a tile in shared memory (rows of 64 features = 128 bytes per chunk,
// 16-byte units XOR-swizzled with the row index).
template <int D>
__device__ __forceinline__ void load_row(uint32_t tile, int r, int lane, float (&x)[D / 32]) {
  constexpr int EPL = D / 32;
  const int e = EPL * lane;                 // first element
  const int c = e / 64;                     // chunk
  const int u = (e % 64) / 8;               // 16-byte unit within the 128-byte row
  const int within = (e % 8) * 2;           // byte offset inside the unit
  const uint32_t addr = tile + c * DecCfg<D>::CHUNK + r * 128 + ((u ^ (r & 7)) << 4) + within;
  if constexpr (EPL == 8) {
    uint32_t a, b, c2, d2;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c2), "=r"(d2)
                 : "r"(addr));
    x[0] = bf_lo(a); x[1] = bf_hi(a); x[2] = bf_lo(b); x[3] = bf_hi(b);
    x[4] = bf_lo(c2); x[5] = bf_hi(c2); x[6] = bf_lo(d2); x[7] = bf_hi(d2);
  } else if constexpr (EPL == 4) {
    uint32_t a, b;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
    x[0] = bf_lo(a); x[1] = bf_hi(a); x[2] = bf_lo(b); x[3] = bf_hi(b);
  } else {
    uint32_t a;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a) : "r"(addr));
    x[0] = bf_lo(a); x[1] = bf_hi(a);
  }
}

template <int D>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecCfg<D>;
  constexpr int EPL = C::EPL;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sK = s_base + C::OFF_K, sV = s_base + C::OFF_V;
  auto full = [&](int s) { return s_base + C::OFF_BAR + 8u * s; };
  auto empty = [&](int s) { return s_base + C::OFF_BAR + 8u * (NS + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);

  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int bh = static_cast<int>(blockIdx.x);
  const int split = static_cast<int>(blockIdx.y);
  const int b = bh / p.H, h = bh % p.H;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kDecWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // global memory only from here on (the set-up may overlap the previous
  // kernel on the stream)
  griddep_wait();
  int n = __ldg(p.cache_lens + b);
  n = n < 0 ? 0 : (n > p.Lk ? p.Lk : n);
  const int k_begin = split * p.chunk;
  const int k_end = min(n, k_begin + p.chunk);
  const int n_tiles = (k_end > k_begin) ? (k_end - k_begin + kDecTile - 1) / kDecTile : 0;

  if (warp == kDecWarps) {
    // ---- TMA warp: K and V tiles of this split into the ring
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      int i = 0;
      for (; i < n_tiles; ++i) {
        const int s = i % NS;
        if (i >= NS && !mbar_wait(empty(s), ((i / NS) - 1) & 1, abort_flag, p.status,
                                  kRoleDecProducer * 64 + s))
          break;
        mbar_arrive_expect_tx(full(s), 2 * C::TILE);
        const int key = k_begin + i * kDecTile;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_4d(sK + s * C::TILE + c * C::CHUNK, &p.tm_k, full(s), 64 * c, h, key, b);
          tma_load_4d(sV + s * C::TILE + c * C::CHUNK, &p.tm_v, full(s), 64 * c, h, key, b);
        }
      }
      // every copy started must land before the CTA exits
      volatile int never = 0;
      for (int t = (i > NS ? i - NS : 0); t < i; ++t)
        mbar_wait(full(t % NS), (t / NS) & 1, &never, p.status, kRoleDecProducer * 64 + 8);
    }
    __syncwarp();
    return;  // no block-wide barrier follows for this warp
  }

  // ---- compute warps
  // q (lane's EPL elements), pre-scaled so that scores come out in log2 units
  // (features past the head's d_k are 0: they add nothing to the scores)
  float qv[EPL];
  {
    const __nv_bfloat16* qrow =
        reinterpret_cast<const __nv_bfloat16*>(p.q) + static_cast<size_t>(bh) * p.d;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int col = EPL * lane + e;
      qv[e] = col < p.d ? __bfloat162float(qrow[col]) * p.scale_log2 : 0.f;
    }
  }
  float m = -INFINITY;       // running maximum of this warp's keys (warp-uniform)
  float l = 0.f;             // running sum; counted in even lanes only
  float acc[EPL];            // unnormalised output, elements EPL*lane ..
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  // After the reduce-scatter below, lane t holds the score of key k = t >> 1.
  const int my_key = lane >> 1;
  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % NS;
    if (!mbar_wait(full(s), (i / NS) & 1, abort_flag, p.status, kRoleDecConsumer * 64 + s)) {
      ok = false;
      break;
    }
    const uint32_t kt = sK + s * C::TILE, vt = sV + s * C::TILE;
    const int r0 = warp * kKeysPerWarp;  // this warp's first row in the tile
    // partial dot products of this lane's elements for the warp's 16 keys
    float v[kKeysPerWarp];
#pragma unroll
    for (int k = 0; k < kKeysPerWarp; ++k) {
      float x[EPL];
      load_row<D>(kt, r0 + k, lane, x);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) d = fmaf(qv[e], x[e], d);
      v[k] = d;
    }
    // reduce-scatter over the lanes: each step halves the values a lane keeps
    // (8, 4, 2, 1 keys) and adds its partner's partial sums for them; the last
    // step completes the sum.  Key k ends in lanes 2k and 2k + 1.
#pragma unroll
    for (int step = 0; step < 4; ++step) {
      const int half = 8 >> step;             // values kept after this step
      const int bit = 16 >> step;             // partner lane distance
      const bool hi = (lane & bit) != 0;      // keep the upper half of the keys
#pragma unroll
      for (int t = 0; t < half; ++t) {
        const float send = hi ? v[t] : v[t + half];
        const float keep = hi ? v[t + half] : v[t];
        v[t] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
      }
    }
    float sc = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
    const int key = k_begin + i * kDecTile + r0 + my_key;
    if (key >= k_end) sc = -INFINITY;         // past this split's keys (or n)
    // online softmax over the warp's keys
    float mt = sc;
#pragma unroll
    for (int o = 2; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    const float m_new = fmaxf(m, mt);
    if (m_new != -INFINITY) {                 // warp-uniform
      const float alpha = ex2_approx(m - m_new);  // 0 on the first keys
      const float pr = ex2_approx(sc - m_new);
      l = l * alpha + ((lane & 1) ? 0.f : pr);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
      m = m_new;
#pragma unroll
      for (int k = 0; k < kKeysPerWarp; ++k) {
        const float pk = __shfl_sync(0xffffffffu, pr, 2 * k);
        float x[EPL];
        load_row<D>(vt, r0 + k, lane, x);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pk, x[e], acc[e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }

  // A CTA that gives up still marks its split's partial as empty (maximum
  // -inf, sum 0), so the combine kernel skips it instead of blending in
  // whatever an earlier call left in the workspace; the status word records
  // the time-out and the output is undefined.
  auto mark_empty = [&]() {
    if (p.n_splits > 1 && lane == 0) {
      p.part_m[static_cast<size_t>(split) * p.B * p.H + bh] = -INFINITY;
      p.part_l[static_cast<size_t>(split) * p.B * p.H + bh] = 0.f;
    }
  };
  // ---- merge the four warps (named barrier 1 over the compute warps only)
  if (!ok) {
    // giving up: let the other compute warps pass the barrier; no output
    mark_empty();
    named_barrier_arrive(1, 32 * kDecWarps);
    return;
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) {
    red[warp] = m;
    red[kDecWarps + warp] = l;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) red[2 * kDecWarps + warp * D + EPL * lane + e] = acc[e];
  named_barrier(1, 32 * kDecWarps);
  if (*abort_flag) {
    mark_empty();
    return;
  }
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red[w]);
  float wgt[kDecWarps];
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) {
    wgt[w] = (red[w] == -INFINITY) ? 0.f : ex2_approx(red[w] - M);
    L += wgt[w] * red[kDecWarps + w];
  }
  // thread t (of the 128) finishes elements t, t + 128, ...
  const int t = static_cast<int>(threadIdx.x);
  if (p.n_splits == 1) {
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(bh) * p.d;
    for (int e = t; e < p.d; e += 32 * kDecWarps) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) o = fmaf(wgt[w], red[2 * kDecWarps + w * D + e], o);
      orow[e] = __float2bfloat16_rn(o * inv);
    }
    if (p.lse && t == 0)
      p.lse[bh] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
  } else {
    float* po = p.part_o + (static_cast<size_t>(split) * p.B * p.H + bh) * D;
    for (int e = t; e < D; e += 32 * kDecWarps) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) o = fmaf(wgt[w], red[2 * kDecWarps + w * D + e], o);
      po[e] = o;
    }
    if (t == 0) {
      p.part_m[static_cast<size_t>(split) * p.B * p.H + bh] = M;
      p.part_l[static_cast<size_t>(split) * p.B * p.H + bh] = L;
    }
  }
}

// One warp per (b, h): merges the split partials into the bf16 output (and lse).
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int EPL = D / 32;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const long long bh = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const long long BH = static_cast<long long>(p.B) * p.H;
  griddep_wait();  // the split kernel's partials are complete and visible
  if (bh >= BH) return;
  float M = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, p.part_m[s * BH + bh]);
  float L = 0.f;
  float o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) o[e] = 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const float ms = p.part_m[s * BH + bh];
    if (ms == -INFINITY) continue;            // a split with no keys
    const float w = ex2_approx(ms - M);
    L = fmaf(w, p.part_l[s * BH + bh], L);
    const float* po = p.part_o + (s * BH + bh) * D + EPL * lane;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, po[e], o[e]);
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + bh * p.d;
#pragma unroll
  for (int e = 0; e < EPL; ++e)
    if (EPL * lane + e < p.d) orow[EPL * lane + e] = __float2bfloat16_rn(o[e] * inv);
  if (p.lse && lane == 0) p.lse[bh] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, cudaStream_t stream, LaunchInfo* info) {
  using C = DecCfg<D>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.n_splits));
  e = launch_serialized(decode_split_kernel<D>, grid, dim3(kDecThreads), C::SMEM, stream, p);
  if (e != cudaSuccess) return e;
  int kernels = 1;
  if (p.n_splits > 1) {
    const long long bh = static_cast<long long>(p.B) * p.H;
    e = launch_serialized(decode_combine_kernel<D>, dim3(static_cast<unsigned>((bh + 7) / 8)),
                          dim3(256), 0, stream, p);
    kernels = 2;
  }
  if (info) {
    info->kernels = kernels;
    info->grid = static_cast<int>(grid.x * grid.y);
    info->block = kDecThreads;
    info->smem = C::SMEM;
  }
  return e;
}

}  // namespace

int decode_splits(int B, int H, int Lk) {
  // enough CTAs for four per SM on a 152-SM part, chunks of at least 256 keys
  const long long bh = static_cast<long long>(B) * H;
  if (bh <= 0 || Lk <= 0) return 1;
  long long s = (608 + bh - 1) / bh;
  const long long by_len = (Lk + kDecChunkMin - 1) / kDecChunkMin;
  if (s > by_len) s = by_len;
  if (s > kDecMaxSplits) s = kDecMaxSplits;
  return s < 1 ? 1 : static_cast<int>(s);
}

int decode_kernel_width(int d) { return d <= 64 ? 64 : (d <= 128 ? 128 : 256); }

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream, LaunchInfo* info) {
  if (p.d < 8 || p.d > 256 || p.d % 8 != 0) return cudaErrorInvalidValue;
  switch (decode_kernel_width(p.d)) {
    case 64: return launch_decode_d<64>(p, stream, info);
    case 128: return launch_decode_d<128>(p, stream, info);
    default: return launch_decode_d<256>(p, stream, info);
  }
}

}  // namespace mha
