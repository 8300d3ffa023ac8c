// kernels.h -- internal launch interface between the C ABI (mha_abi.cu) and
// the kernels.  Not installed; no torch or Python types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace mha {

// Mask kinds are bit sets: kMaskCausalKeyPadding applies both masks.
enum MaskKind : int { kMaskNone = 0, kMaskCausal = 1, kMaskKeyPadding = 2, kMaskCausalKeyPadding = 3 };
__host__ __device__ __forceinline__ bool masks_causal(int mask_kind) { return (mask_kind & kMaskCausal) != 0; }
__host__ __device__ __forceinline__ bool masks_padding(int mask_kind) { return (mask_kind & kMaskKeyPadding) != 0; }

// Queries per tile (M of the tcgen05 MMA), keys per K/V tile, and query rows
// per work unit of the bf16 kernel (two tiles share every K/V tile).
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kUnitRows = 2 * kBlockM;

struct Bf16Params {
  CUtensorMap tm_q;  // [B, Lq, H, d] bf16, box {64, 1, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k;  // [B, Lk, H, d]
  CUtensorMap tm_v;  // [B, Lk, H, d]
  CUtensorMap tm_o;  // [B, Lq, H, d] bf16 output, same box and swizzle as tm_q
  void* out;         // [B, Lq, H, d] bf16
  float* lse;        // [B, H, Lq] natural-log log-sum-exp per row, or null
  const int32_t* key_lens;
  DeviceStatus* status;
  int B, H, Lq, Lk;
  int mask_kind;
  int n_qtiles;      // query blocks per head: ceil(Lq / kUnitRows); the launch
                     // sets ceil(Lq / kBlockM) when it pairs heads
  int head_group;    // set by the launch: heads whose units are dispatched
                     // together (their K/V stay in L2); even
  int paired;        // set by the launch: 0 = a unit is two query tiles of one
                     // head sharing every K/V tile; 1 (d_k = 64) = a unit is the
                     // same query tile of two heads, each with its own K/V tiles
  float scale_log2;  // scale * log2(e)
  int dk_steps;      // K16 steps of S = Q K^T: ceil(d_k / 16) <= D / 16
  int dv_n;          // N of the P.V products: d_v rounded up to 16, <= D
  int withhold_p;    // test hook: softmax 0 withholds its first P arrival (0 = off)
};

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;        // [B, H, Lq] natural-log log-sum-exp per row, or null
  const int32_t* key_lens;
  int B, H, Lq, Lk, d;  // d: width of q and k rows (d_k)
  int dv;               // width of v and output rows (d_v)
  int mask_kind;
  float scale_log2;
};

struct LaunchInfo {
  int kernels = 0;
  int grid = 0;
  int block = 0;
  int smem = 0;
};

// Decode step: one query row per (sequence, head) against a key/value cache.
struct DecodeParams {
  CUtensorMap tm_k;  // [B, Lk, H, d] bf16 cache, box {64, 1, 64, 1}, 128-byte swizzle
  CUtensorMap tm_v;
  const void* q;     // [B, H, d] bf16
  void* out;         // [B, H, d] bf16
  float* lse;        // [B, H] or null
  const int32_t* cache_lens;  // [B] keys per sequence (clamped to [0, Lk])
  float* part_o;     // [n_splits, B*H, kernel width]  (n_splits > 1)
  float* part_m;     // [n_splits, B*H]
  float* part_l;     // [n_splits, B*H]
  DeviceStatus* status;
  int B, H, Lk;
  int d;             // head width d_k: a multiple of 8 up to 256 (the kernel's
                     // width, 64, 128 or 256, is the next one up)
  int chunk;         // keys per split, a multiple of 64
  int n_splits;
  float scale_log2;  // scale * log2(e)
};

constexpr int kDecChunkMin = 256;   // fewest keys a split is given
constexpr int kDecMaxSplits = 64;

// Splits the decode kernel uses for these sizes (the workspace holds that many
// partial results unless it is 1).
int decode_splits(int B, int H, int Lk);

// Width of the decode kernel a head of d features runs on (64, 128 or 256).
int decode_kernel_width(int d);

// Launches the decode step (p.d a multiple of 8 up to 256): the split kernel
// and, with more than one split, the combine kernel.
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream, LaunchInfo* info);

// Gradient of the bf16 forward.
struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // [B, L, H, d] bf16, box {64, 1, 128, 1}, 128-byte swizzle
  CUtensorMap tm_o;                      // [B, Lq, H, d] the forward output, same box
  CUtensorMap tm_dk, tm_dv;              // [B, Lk, H, d] the key gradients (stored), same box
  const void* out;    // [B, Lq, H, d] bf16 forward output
  const void* dout;   // [B, Lq, H, d] bf16 dL/dO
  const float* lse;   // [B, H, Lq] forward row log-sum-exp (natural log)
  float* dvec;        // [B, H, Lq] workspace: D_i = dO_i . O_i
  void* dq;           // [B, Lq, H, d] bf16
  void* dk;           // [B, Lk, H, d] bf16
  void* dv;           // [B, Lk, H, d] bf16
  const int32_t* key_lens;
  DeviceStatus* status;
  int B, H, Lq, Lk;
  int d;              // row width of q, k, v, out and the gradients (a multiple of 8,
                      // at most the kernel's width; the tensor maps zero-fill the rest)
  int mask_kind;
  float scale;        // multiplier of q . k
  float scale_log2;   // scale * log2(e)
  int head_group;     // set by the launch: heads whose units are dispatched together
};

// Launches the gradient: the dQ kernel (which also forms D) and the dK/dV kernel.
cudaError_t launch_bwd(const BwdParams& p, int d, cudaStream_t stream, LaunchInfo* info);

// Launches the bf16 tcgen05 forward for d in {64, 128}.
cudaError_t launch_fwd_bf16(const Bf16Params& p, int d, cudaStream_t stream, LaunchInfo* info);

// Launches the one-query-tile bf16 tcgen05 forward (mha_fwd_wide.cu) at
// width 256 (heads wider than 128, d_k and d_v up to 256) or 64 (the light
// variant, two CTAs per SM, for short sequences of heads up to 64 wide):
// tm_q box {64, 1, 128, 1}, tm_k and tm_v box {64, 1, 64, 1}, tm_o box
// {64, 1, 32, 1}; sets n_qtiles and head_group.
cudaError_t launch_fwd_wide(const Bf16Params& p, int width, cudaStream_t stream, LaunchInfo* info);

// Launches a kernel with programmatic stream serialization: its grid may be
// scheduled while the previous kernel on the stream drains, so its set-up
// overlaps that kernel's tail.  The kernel must call griddep_wait() before
// its first global memory access.
template <typename... Params, typename... Args>
inline cudaError_t launch_serialized(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Launches the float32 SIMT forward (1 <= d <= 256).
cudaError_t launch_fwd_f32(const F32Params& p, cudaStream_t stream, LaunchInfo* info);

// Row-major bf16 GEMM on the tensor cores (mha_gemm.cu): C[M x N] =
// A[M x K] B[K x N], float32 accumulation, bf16 result.
struct GemmParams {
  CUtensorMap tm_a;  // A [M, K] (row stride lda), box {64 k, 128 rows}, 128-byte swizzle
  CUtensorMap tm_b;  // B [K, N] (row stride ldb), box {64 n, 64 k}, 128-byte swizzle
  CUtensorMap tm_c;  // C [M, N] (row stride ldc), box {64 n, 32 rows}, 128-byte swizzle
  DeviceStatus* status;
  int M, N, K;
  int tiles_m, tiles_n;  // set by the launch: row blocks (128 or 256 rows), ceil(N / 256)
  int k_blocks;          // set by the launch: ceil(K / 64)
};

// Launches the GEMM (one persistent CTA per SM, or per tile when fewer; tiles
// of 128 x 256, or 256 x 256 when K is long); adds one to info->kernels.
cudaError_t launch_gemm(const GemmParams& p, cudaStream_t stream, LaunchInfo* info);

}  // namespace mha
