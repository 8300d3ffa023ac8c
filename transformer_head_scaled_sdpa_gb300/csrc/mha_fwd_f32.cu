// mha_fwd_f32.cu -- float32 attention forward on the CUDA cores.
//
// The same operation as the bf16 path ("Attention Is All You Need",
// Section 3.2.1, Equation (1), every head in parallel), all in float32, for
// any head size 1 <= d_k, d_v <= 256 (d_v, the value width, may differ from
// d_k).  One warp owns one query row (b, i, h):
//   - q (pre-multiplied by scale * log2(e)) is staged in shared memory;
//   - keys are visited 32 at a time, one per lane: lane t scores key j0 + t;
//   - the online softmax keeps a running maximum m and sum l per row and
//     rescales the partial output by 2^(m_old - m_new) when m grows (exact,
//     by the shift invariance of the weights: formula page
//     transformer-attention, section 証明);
//   - each lane accumulates output components lane, lane + 32, ... over the
//     32 keys, whose weights are broadcast with shuffles, so V rows are read
//     coalesced.
// Masks remove keys before the softmax: causal keeps keys j <= i, key padding
// keeps j < key_lens[b] (clamped to [0, Lk]), both together keep keys that
// pass both.  A row with no key stores 0.
// Optionally each row's log-sum-exp (the log of the softmax denominator) is
// stored as well; -inf for a row with no key.
#include "kernels.h"

namespace mha {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxD = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) fwd_f32_kernel(const F32Params p) {
  extern __shared__ float s_q[];  // kWarpsPerBlock x d
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const long long rows = static_cast<long long>(p.B) * p.H * p.Lq;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + warp;
  if (row >= rows) return;  // whole warp leaves together; no block barrier below

  // row enumerates (b, i, h) with h fastest, matching the [B, Lq, H, d] layout
  const int h = static_cast<int>(row % p.H);
  const int i = static_cast<int>((row / p.H) % p.Lq);
  const int b = static_cast<int>(row / (static_cast<long long>(p.H) * p.Lq));
  const int d = p.d, dv = p.dv;

  int n = p.Lk;
  if (masks_causal(p.mask_kind)) n = (i + 1 < p.Lk) ? i + 1 : p.Lk;
  if (masks_padding(p.mask_kind)) {
    const int len = __ldg(p.key_lens + b);
    const int clamped = len < 0 ? 0 : (len > p.Lk ? p.Lk : len);
    if (clamped < n) n = clamped;
  }

  float* q_s = s_q + warp * d;
  const float* q_row = p.q + (static_cast<size_t>(row)) * d;  // (b*Lq + i)*H + h == row
  for (int c = lane; c < d; c += 32) q_s[c] = q_row[c] * p.scale_log2;
  __syncwarp();

  const size_t kv_stride = static_cast<size_t>(p.H) * d;   // between consecutive keys
  const size_t v_stride = static_cast<size_t>(p.H) * dv;   // between consecutive value rows
  const float* k_bh = p.k + (static_cast<size_t>(b) * p.Lk * p.H + h) * d;
  const float* v_bh = p.v + (static_cast<size_t>(b) * p.Lk * p.H + h) * dv;

  constexpr int kPerLane = kMaxD / 32;
  float acc[kPerLane];
#pragma unroll
  for (int t = 0; t < kPerLane; ++t) acc[t] = 0.f;
  float m = -INFINITY;
  float l = 0.f;

  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    float s = -INFINITY;
    if (j < n) {
      const float* k_row = k_bh + static_cast<size_t>(j) * kv_stride;
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(q_s[c], k_row[c], dot);
      s = dot;  // already in log2 units
    }
    const float m_new = fmaxf(m, warp_max(s));   // finite: lane 0 holds a key
    const float alpha = exp2f(m - m_new);        // 0 on the first chunk
    const float pj = (j < n) ? exp2f(s - m_new) : 0.f;
    l = l * alpha + warp_sum(pj);
    m = m_new;
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) acc[t] *= alpha;
    const int cnt = (n - j0 < 32) ? (n - j0) : 32;
    for (int t = 0; t < cnt; ++t) {
      const float pt = __shfl_sync(0xffffffffu, pj, t);
      const float* v_row = v_bh + static_cast<size_t>(j0 + t) * v_stride;
#pragma unroll
      for (int u = 0; u < kPerLane; ++u) {
        const int c = lane + 32 * u;
        if (c < dv) acc[u] = fmaf(pt, v_row[c], acc[u]);
      }
    }
  }

  float* o_row = p.out + static_cast<size_t>(row) * dv;
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  if (p.lse && lane == 0) {
    // log of the softmax denominator, natural units: m and the exponents are
    // in log2 units of the scaled scores, so lse = (m + log2 l) * ln 2
    p.lse[(static_cast<size_t>(b) * p.H + h) * p.Lq + i] =
        (l > 0.f) ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
#pragma unroll
  for (int u = 0; u < kPerLane; ++u) {
    const int c = lane + 32 * u;
    if (c < dv) o_row[c] = acc[u] * inv;
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const F32Params& p, cudaStream_t stream, LaunchInfo* info) {
  if (p.d < 1 || p.d > kMaxD || p.dv < 1 || p.dv > kMaxD) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(p.B) * p.H * p.Lq;
  const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int smem = kWarpsPerBlock * p.d * static_cast<int>(sizeof(float));
  fwd_f32_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, smem, stream>>>(p);
  if (info) {
    info->kernels = 1;
    info->grid = static_cast<int>(blocks);
    info->block = kWarpsPerBlock * 32;
    info->smem = smem;
  }
  return cudaGetLastError();
}

}  // namespace mha
