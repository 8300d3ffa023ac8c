// mha_abi.cu -- the C ABI of libmha.so (declared in include/mha.h, its test
// hooks in include/mha_test_hooks.h): argument
// checks, TMA tensor-map encoding, kernel dispatch, the host-buffer entry and
// the per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mha.h"
#include "../../include/mha_test_hooks.h"
#include "kernels.h"

namespace {

using mha::DeviceStatus;

// One status word per device: kernels record a bounded wait that gave up.
__device__ DeviceStatus g_status;

// Scratch of mha_decode_static (the split partials of one decode step), for
// callers that pass no workspace: 2 MiB per device, shared by every call of
// that entry on the device.
constexpr size_t kDecodeStaticScratchBytes = size_t(2) << 20;
static __device__ __align__(256) uint8_t g_decode_scratch[kDecodeStaticScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int supported = 0;  // MHA_OK or MHA_ERR_UNSUPPORTED
  DeviceStatus* status = nullptr;
  void* decode_scratch = nullptr;  // device address of g_decode_scratch
};

std::mutex g_mutex;
int g_withhold_p = 0;  // test hook of mha_debug_withhold_p
DeviceState g_dev[kMaxDevices];

// The host entry's two streams and its events, created on the device's
// first mha_fwd_host call and kept for the process.  `order` is held while a
// call records `start` and queues its chunks, so two host threads calling at
// once cannot re-record each other's start event (the internal streams would
// then wait on the other caller's stream) or interleave chunks on the shared
// streams.
struct HostPipe {
  bool ready = false;
  cudaStream_t st[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr, done[2] = {nullptr, nullptr};
  std::mutex order;
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return MHA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    for (int i = 0; i < 2; ++i) {
      if (!hp.st[i] && cudaStreamCreateWithFlags(&hp.st[i], cudaStreamNonBlocking) != cudaSuccess)
        return MHA_ERR_LAUNCH;
      if (!hp.done[i] &&
          cudaEventCreateWithFlags(&hp.done[i], cudaEventDisableTiming) != cudaSuccess)
        return MHA_ERR_LAUNCH;
    }
    if (!hp.start && cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) != cudaSuccess)
      return MHA_ERR_LAUNCH;
    hp.ready = true;
  }
  *out = &hp;
  return MHA_OK;
}
thread_local mha::LaunchInfo t_info;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Device set-up, once per device with that device current: capability check
// and the device address of the status word.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return MHA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MHA_ERR_LAUNCH;
    st.supported = (major == 10 && minor == 3) ? MHA_OK : MHA_ERR_UNSUPPORTED;
    if (st.supported == MHA_OK) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) return MHA_ERR_LAUNCH;
      st.status = static_cast<DeviceStatus*>(addr);
      if (cudaGetSymbolAddress(&st.decode_scratch, g_decode_scratch) != cudaSuccess)
        return MHA_ERR_LAUNCH;
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
          return MHA_ERR_LAUNCH;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    st.ready = true;
  }
  *out = &st;
  return st.supported;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a);
  const uintptr_t y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

struct Sizes {
  size_t q_elems = 0, kv_elems = 0;  // q (and k) rows of d_k elements
  size_t v_elems = 0, o_elems = 0;   // v and out rows of d_v elements
};

bool mask_known(int mask_kind) {
  return mask_kind >= MHA_MASK_NONE && mask_kind <= MHA_MASK_CAUSAL_KEY_PADDING;
}
bool has_causal(int mask_kind) { return (mask_kind & MHA_MASK_CAUSAL) != 0; }
bool has_padding(int mask_kind) { return (mask_kind & MHA_MASK_KEY_PADDING) != 0; }

// Checks shared by the device entries (d_v: the width of v and out rows).
// Returns MHA_OK and sets *empty when there is nothing to compute.
int check_args(const void* q, const void* k, const void* v, void* out, int B, int H, int Lq,
               int Lk, int d_k, int d_v, int mask_kind, const int32_t* key_lens, float scale,
               int elem_bytes, size_t align, bool* empty, Sizes* sz) {
  *empty = false;
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || d_k < 0 || d_v < 0) return MHA_ERR_SHAPE;
  if (!mask_known(mask_kind)) return MHA_ERR_MASK;
  if (has_causal(mask_kind) && Lq != Lk) return MHA_ERR_SHAPE;
  if (!std::isfinite(scale) || scale < 0.f) return MHA_ERR_SCALE;
  if (d_k == 0 || d_v == 0) return MHA_ERR_SHAPE;
  // every element index must fit comfortably in 64 bits and every row count in 31
  const long long rows_q = static_cast<long long>(B) * H * Lq;
  const long long rows_k = static_cast<long long>(B) * H * Lk;
  if (rows_q > (1ll << 40) || rows_k > (1ll << 40)) return MHA_ERR_SHAPE;
  sz->q_elems = static_cast<size_t>(rows_q) * d_k;
  sz->kv_elems = static_cast<size_t>(rows_k) * d_k;
  sz->v_elems = static_cast<size_t>(rows_k) * d_v;
  sz->o_elems = static_cast<size_t>(rows_q) * d_v;
  if (rows_q == 0) {
    *empty = true;
    return MHA_OK;
  }
  if (!q || !out) return MHA_ERR_NULL;
  if (Lk > 0 && (!k || !v)) return MHA_ERR_NULL;
  if (has_padding(mask_kind) && !key_lens) return MHA_ERR_MASK;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                         (Lk > 0 ? (reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v))
                                 : 0)) &
                        (align - 1);
  if (mis) return MHA_ERR_UNSUPPORTED;
  const size_t ob = sz->o_elems * elem_bytes;
  if (overlaps(out, ob, q, sz->q_elems * elem_bytes) ||
      overlaps(out, ob, k, sz->kv_elems * elem_bytes) ||
      overlaps(out, ob, v, sz->v_elems * elem_bytes))
    return MHA_ERR_ALIAS;
  return MHA_OK;
}

// bf16 rows on the tensor-core kernels: a multiple of 8 elements (16-byte row
// strides for the tensor maps) up to 256 for the forward (128 for the
// gradient); narrower rows are zero-filled by the tensor-map loads up to the
// kernel's width (64, 128, or 256 on the wide kernel) and clipped on store.
bool bf16_width_ok(int d) { return d >= 8 && d <= 256 && d % 8 == 0; }
bool bf16_bwd_width_ok(int d) { return d >= 8 && d <= 128 && d % 8 == 0; }
int bf16_kernel_width(int d_k, int d_v) {
  return (d_k <= 64 && d_v <= 64) ? 64 : ((d_k <= 128 && d_v <= 128) ? 128 : 256);
}

// 4-D map over a [B, L, H, d] bf16 tensor; box = 64 features x 1 head x `rows`
// rows (128 for the forward's tiles, 64 for the decode step's) x 1 sequence,
// 128-byte swizzle (the tcgen05 operand layout).  Features past d read as 0
// and are not written by stores.
// row_elems: elements between consecutive positions of one head (H*d for a
// dense tensor; more when the rows interleave other tensors, as the packed
// Q|K|V projection output does).
bool encode_map(CUtensorMap* m, const void* base, int B, int L, int H, int d, int rows = 128,
                long long row_elems = -1) {
  if (row_elems < 0) row_elems = static_cast<long long>(H) * d;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(row_elems) * 2,
                                 static_cast<cuuint64_t>(L) * row_elems * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr float kLog2e = 1.4426950408889634f;

// lse, when requested: [B, H, Lq] float32, 4-byte aligned, overlapping none of
// q, k, v, out.
int check_lse(const float* lse, const void* q, const void* k, const void* v, const void* out,
              const Sizes& sz, int elem_bytes, long long rows_q) {
  if (!lse) return MHA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return MHA_ERR_UNSUPPORTED;
  const size_t lb = static_cast<size_t>(rows_q) * 4;
  if (overlaps(lse, lb, q, sz.q_elems * elem_bytes) ||
      overlaps(lse, lb, out, sz.o_elems * elem_bytes) ||
      overlaps(lse, lb, k, sz.kv_elems * elem_bytes) ||
      overlaps(lse, lb, v, sz.v_elems * elem_bytes))
    return MHA_ERR_ALIAS;
  return MHA_OK;
}

__global__ void fill_f32_kernel(float* p, size_t n, float value) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = value;
}

// With no key anywhere every output row is 0 and every lse -inf.
int no_keys(void* out, size_t out_bytes, float* lse, size_t rows, cudaStream_t s) {
  if (cudaMemsetAsync(out, 0, out_bytes, s) != cudaSuccess) return MHA_ERR_LAUNCH;
  if (lse) {
    const unsigned blocks = static_cast<unsigned>(rows < 256 * 1024 ? (rows + 255) / 256 : 1024);
    fill_f32_kernel<<<blocks, 256, 0, s>>>(lse, rows, -INFINITY);
    if (cudaGetLastError() != cudaSuccess) return MHA_ERR_LAUNCH;
    t_info.kernels = 1;
    t_info.grid = static_cast<int>(blocks);
    t_info.block = 256;
  }
  return MHA_OK;
}

// One CTA waits on an mbarrier that nothing ever arrives on, with the same
// bounded wait the pipelines use: after the limit it records
// MHA_ERR_TIMEOUT in the status word and returns.
__global__ void selftest_wait_kernel(DeviceStatus* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mha::mbar_init(mha::smem_u32(&bar), 1);
    abort_flag = 0;
    mha::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mha::mbar_wait(mha::smem_u32(&bar), 0, &abort_flag, status, 0xFF);
  __syncthreads();
}

float effective_scale(float scale, int d_k) {
  return scale == 0.f ? 1.f / std::sqrt(static_cast<float>(d_k)) : scale;
}

int attention_bf16(const void* q, const void* k, const void* v, void* out, float* lse,
                   long long q_row, long long k_row, long long v_row, int B, int H, int Lq,
                   int Lk, int d_k, int d_v, int mask_kind, const int32_t* key_lens, float scale,
                   DeviceState* dev, cudaStream_t s);

int fwd_bf16(const void* q, const void* k, const void* v, void* out, float* lse, bool want_lse,
             int B, int H, int Lq, int Lk, int d_k, int d_v, int mask_kind,
             const int32_t* key_lens, float scale, void* stream) {
  t_info = mha::LaunchInfo{};
  bool empty = false;
  Sizes sz;
  int rc = check_args(q, k, v, out, B, H, Lq, Lk, d_k, d_v, mask_kind, key_lens, scale, 2, 16,
                      &empty, &sz);
  if (rc != MHA_OK) return rc;
  if (!bf16_width_ok(d_k) || !bf16_width_ok(d_v)) return MHA_ERR_UNSUPPORTED;
  if (empty) return MHA_OK;
  const long long rows_q = static_cast<long long>(B) * H * Lq;
  if (want_lse && (rc = check_lse(lse, q, k, v, out, sz, 2, rows_q)) != MHA_OK) return rc;
  DeviceState* dev = nullptr;
  rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Lk == 0) return no_keys(out, sz.o_elems * 2, lse, static_cast<size_t>(rows_q), s);
  return attention_bf16(q, k, v, out, lse, static_cast<long long>(H) * d_k,
                        static_cast<long long>(H) * d_k, static_cast<long long>(H) * d_v, B, H,
                        Lq, Lk, d_k, d_v, mask_kind, key_lens, scale, dev, s);
}

// Heads up to 64 wide over short sequences without the causal mask take the
// light one-tile kernel (two CTAs per SM, so one CTA's unit boundary overlaps
// another's tiles).  Measured against the two-tile kernel, graph-timed with
// the inputs out of L2: -7 % on 32 x 8 heads at L 128, the same at Lq 256 /
// Lk 512 with key padding, +5 % under the causal mask at L 512 (there the
// two-tile kernel's shared K/V tiles win).
static bool light_forward(int Lq, int Lk, int mask_kind) {
  return Lq <= 512 && Lk <= 512 && (mask_kind & MHA_MASK_CAUSAL) == 0;
}

// The bf16 attention launch on checked arguments (Lq, Lk > 0).  q_row, k_row,
// v_row: elements between consecutive positions of one head in q, k, v; out is
// dense [B, Lq, H, d_v].
int attention_bf16(const void* q, const void* k, const void* v, void* out, float* lse,
                   long long q_row, long long k_row, long long v_row, int B, int H, int Lq,
                   int Lk, int d_k, int d_v, int mask_kind, const int32_t* key_lens, float scale,
                   DeviceState* dev, cudaStream_t s) {
  const long long n_qtiles = (Lq + mha::kUnitRows - 1) / mha::kUnitRows;
  if (n_qtiles * B * H > 0x7fffffffll) return MHA_ERR_SHAPE;
  mha::Bf16Params p;
  std::memset(&p, 0, sizeof(p));
  // the one-tile kernel (heads wider than 128; short sequences of heads up to
  // 64 wide) streams 64-key tiles and each epilogue warp stores its own 32 rows
  const int width = bf16_kernel_width(d_k, d_v);
  const bool wide = width > 128;
  const bool light = width == 64 && light_forward(Lq, Lk, mask_kind);
  const bool one_tile = wide || light;
  if (!encode_map(&p.tm_q, q, B, Lq, H, d_k, 128, q_row) ||
      !encode_map(&p.tm_k, k, B, Lk, H, d_k, one_tile ? 64 : 128, k_row) ||
      !encode_map(&p.tm_v, v, B, Lk, H, d_v, one_tile ? 64 : 128, v_row) ||
      !encode_map(&p.tm_o, out, B, Lq, H, d_v, one_tile ? 32 : 128))
    return MHA_ERR_UNSUPPORTED;
  p.out = out;
  p.lse = lse;
  p.key_lens = key_lens;
  p.status = dev->status;
  p.B = B;
  p.H = H;
  p.Lq = Lq;
  p.Lk = Lk;
  p.mask_kind = mask_kind;
  p.n_qtiles = static_cast<int>(n_qtiles);
  p.scale_log2 = effective_scale(scale, d_k) * kLog2e;
  p.dk_steps = (d_k + 15) / 16;
  p.dv_n = (d_v + 15) / 16 * 16;
  p.withhold_p = g_withhold_p;
  const cudaError_t e = one_tile ? mha::launch_fwd_wide(p, wide ? 256 : 64, s, &t_info)
                                 : mha::launch_fwd_bf16(p, width, s, &t_info);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_LAUNCH;
}

int fwd_f32(const void* q, const void* k, const void* v, void* out, float* lse, bool want_lse,
            int B, int H, int Lq, int Lk, int d_k, int d_v, int mask_kind,
            const int32_t* key_lens, float scale, void* stream) {
  t_info = mha::LaunchInfo{};
  bool empty = false;
  Sizes sz;
  int rc = check_args(q, k, v, out, B, H, Lq, Lk, d_k, d_v, mask_kind, key_lens, scale, 4, 4,
                      &empty, &sz);
  if (rc != MHA_OK) return rc;
  if (d_k > 256 || d_v > 256) return MHA_ERR_UNSUPPORTED;
  if (empty) return MHA_OK;
  const long long rows_q = static_cast<long long>(B) * H * Lq;
  if (want_lse && (rc = check_lse(lse, q, k, v, out, sz, 4, rows_q)) != MHA_OK) return rc;
  DeviceState* dev = nullptr;
  rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Lk == 0) return no_keys(out, sz.o_elems * 4, lse, static_cast<size_t>(rows_q), s);
  if ((static_cast<long long>(B) * H * Lq + 7) / 8 > 0x7fffffffll) return MHA_ERR_SHAPE;
  mha::F32Params p;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.out = static_cast<float*>(out);
  p.lse = lse;
  p.key_lens = key_lens;
  p.B = B;
  p.H = H;
  p.Lq = Lq;
  p.Lk = Lk;
  p.d = d_k;
  p.dv = d_v;
  p.mask_kind = mask_kind;
  p.scale_log2 = effective_scale(scale, d_k) * kLog2e;
  return mha::launch_fwd_f32(p, s, &t_info) == cudaSuccess ? MHA_OK : MHA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int mha_fwd(const void* q, const void* k, const void* v, void* out, int B, int H, int Lq, int Lk,
            int d_k, int mask_kind, const int32_t* key_lens, float scale, void* stream) {
  return fwd_bf16(q, k, v, out, nullptr, false, B, H, Lq, Lk, d_k, d_k, mask_kind, key_lens,
                  scale, stream);
}

int mha_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                int Lq, int Lk, int d_k, int mask_kind, const int32_t* key_lens, float scale,
                void* stream) {
  return fwd_bf16(q, k, v, out, lse, true, B, H, Lq, Lk, d_k, d_k, mask_kind, key_lens, scale,
                  stream);
}

int mha_fwd_dv(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
               int Lq, int Lk, int d_k, int d_v, int mask_kind, const int32_t* key_lens,
               float scale, void* stream) {
  return fwd_bf16(q, k, v, out, lse, lse != nullptr, B, H, Lq, Lk, d_k, d_v, mask_kind, key_lens,
                  scale, stream);
}

int mha_fwd_f32(const void* q, const void* k, const void* v, void* out, int B, int H, int Lq,
                int Lk, int d_k, int mask_kind, const int32_t* key_lens, float scale,
                void* stream) {
  return fwd_f32(q, k, v, out, nullptr, false, B, H, Lq, Lk, d_k, d_k, mask_kind, key_lens, scale,
                 stream);
}

int mha_fwd_f32_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int H, int Lq, int Lk, int d_k, int mask_kind, const int32_t* key_lens,
                    float scale, void* stream) {
  return fwd_f32(q, k, v, out, lse, true, B, H, Lq, Lk, d_k, d_k, mask_kind, key_lens, scale,
                 stream);
}

int mha_fwd_f32_dv(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                   int H, int Lq, int Lk, int d_k, int d_v, int mask_kind,
                   const int32_t* key_lens, float scale, void* stream) {
  return fwd_f32(q, k, v, out, lse, lse != nullptr, B, H, Lq, Lk, d_k, d_v, mask_kind, key_lens,
                 scale, stream);
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace of the decode step: partial outputs, maxima and sums of every
// split (none with a single split).
// (partial outputs are kept at the kernel's width: 64, 128 or 256)
static size_t decode_ws_bytes(int B, int H, int Lk, int d_k, int* splits_out) {
  const int S = mha::decode_splits(B, H, Lk);
  if (splits_out) *splits_out = S;
  if (S <= 1) return 0;
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t w = static_cast<size_t>(mha::decode_kernel_width(d_k));
  return align256(static_cast<size_t>(S) * bh * w * 4) + 2 * align256(static_cast<size_t>(S) * bh * 4);
}

// decode head widths: multiples of 8 from 8 to 256
static bool decode_width_ok(int d) { return d >= 8 && d <= 256 && d % 8 == 0; }

size_t mha_decode_workspace_bytes(int B, int H, int Lk, int d_k) {
  if (B < 0 || H < 0 || Lk < 0 || !decode_width_ok(d_k)) return 0;
  return decode_ws_bytes(B, H, Lk, d_k, nullptr);
}

// The decode step with the split partials in `workspace` (from the caller) or,
// with use_static, in this device's static scratch.
static int decode_step(const void* q, const void* k_cache, const void* v_cache, void* out,
                       float* lse, int B, int H, int Lk, int d_k, const int32_t* cache_lens,
                       float scale, void* workspace, size_t workspace_bytes, bool use_static,
                       void* stream) {
  t_info = mha::LaunchInfo{};
  if (B < 0 || H < 0 || Lk < 0) return MHA_ERR_SHAPE;
  if (!std::isfinite(scale) || scale < 0.f) return MHA_ERR_SCALE;
  if (!decode_width_ok(d_k)) return MHA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  const long long cache_rows = bh * Lk;
  if (bh > 0x7fffffffll || cache_rows > (1ll << 40)) return MHA_ERR_SHAPE;
  if (bh == 0) return MHA_OK;
  if (!q || !out) return MHA_ERR_NULL;
  if (!cache_lens) return MHA_ERR_MASK;
  if (Lk > 0 && (!k_cache || !v_cache)) return MHA_ERR_NULL;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
                         (Lk > 0 ? (reinterpret_cast<uintptr_t>(k_cache) |
                                    reinterpret_cast<uintptr_t>(v_cache))
                                 : 0)) &
                        15u;
  if (mis || (reinterpret_cast<uintptr_t>(lse) & 3u)) return MHA_ERR_UNSUPPORTED;
  const size_t qb = static_cast<size_t>(bh) * d_k * 2;
  const size_t kb = static_cast<size_t>(cache_rows) * d_k * 2;
  const size_t lb = static_cast<size_t>(bh) * 4;
  if (overlaps(out, qb, q, qb) || overlaps(out, qb, k_cache, kb) || overlaps(out, qb, v_cache, kb))
    return MHA_ERR_ALIAS;
  if (lse && (overlaps(lse, lb, out, qb) || overlaps(lse, lb, q, qb) ||
              overlaps(lse, lb, k_cache, kb) || overlaps(lse, lb, v_cache, kb)))
    return MHA_ERR_ALIAS;
  int S = 1;
  const size_t need = decode_ws_bytes(B, H, Lk, d_k, &S);
  if (use_static) {
    if (need > kDecodeStaticScratchBytes) return MHA_ERR_WORKSPACE;
  } else {
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 15u)))
      return MHA_ERR_WORKSPACE;
    if (need > 0 && overlaps(workspace, need, out, qb)) return MHA_ERR_ALIAS;
  }
  DeviceState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  if (use_static) workspace = dev->decode_scratch;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Lk == 0) return no_keys(out, qb, lse, static_cast<size_t>(bh), s);
  mha::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_map(&p.tm_k, k_cache, B, Lk, H, d_k, 64) ||
      !encode_map(&p.tm_v, v_cache, B, Lk, H, d_k, 64))
    return MHA_ERR_UNSUPPORTED;
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.cache_lens = cache_lens;
  if (S > 1) {
    // every split CTA writes its whole partial (an empty split: output 0,
    // maximum -inf, sum 0) before the combine reads it: nothing starts at zero
    uint8_t* w = static_cast<uint8_t*>(workspace);
    p.part_o = reinterpret_cast<float*>(w);
    w += align256(static_cast<size_t>(S) * bh * mha::decode_kernel_width(d_k) * 4);
    p.part_m = reinterpret_cast<float*>(w);
    w += align256(static_cast<size_t>(S) * bh * 4);
    p.part_l = reinterpret_cast<float*>(w);
  }
  p.status = dev->status;
  p.B = B;
  p.H = H;
  p.Lk = Lk;
  p.d = d_k;
  p.n_splits = S;
  const int per = (Lk + S - 1) / S;
  p.chunk = (per + 63) / 64 * 64;
  p.scale_log2 = effective_scale(scale, d_k) * kLog2e;
  return mha::launch_decode(p, s, &t_info) == cudaSuccess ? MHA_OK : MHA_ERR_LAUNCH;
}

int mha_decode(const void* q, const void* k_cache, const void* v_cache, void* out, float* lse,
               int B, int H, int Lk, int d_k, const int32_t* cache_lens, float scale,
               void* workspace, size_t workspace_bytes, void* stream) {
  return decode_step(q, k_cache, v_cache, out, lse, B, H, Lk, d_k, cache_lens, scale, workspace,
                     workspace_bytes, false, stream);
}

int mha_decode_static(const void* q, const void* k_cache, const void* v_cache, void* out,
                      float* lse, int B, int H, int Lk, int d_k, const int32_t* cache_lens,
                      float scale, void* stream) {
  return decode_step(q, k_cache, v_cache, out, lse, B, H, Lk, d_k, cache_lens, scale, nullptr, 0,
                     true, stream);
}

size_t mha_decode_static_scratch_bytes(void) { return kDecodeStaticScratchBytes; }

size_t mha_bwd_workspace_bytes(int B, int H, int Lq, int Lk, int d_k) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || !bf16_bwd_width_ok(d_k)) return 0;
  return align256(static_cast<size_t>(B) * H * Lq * 4);
}

int mha_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
            const float* lse, void* dq, void* dk, void* dv, int B, int H, int Lq, int Lk,
            int d_k, int mask_kind, const int32_t* key_lens, float scale, void* workspace,
            size_t workspace_bytes, void* stream) {
  t_info = mha::LaunchInfo{};
  bool empty = false;
  Sizes sz;
  // the forward's checks on q, k, v, out (and the mask, scale, sizes)
  int rc = check_args(q, k, v, const_cast<void*>(out), B, H, Lq, Lk, d_k, d_k, mask_kind,
                      key_lens, scale, 2, 16, &empty, &sz);
  if (rc != MHA_OK) return rc;
  if (!bf16_bwd_width_ok(d_k)) return MHA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0) return MHA_OK;
  const size_t qb = sz.q_elems * 2, kb = sz.kv_elems * 2;
  const size_t lb = static_cast<size_t>(bh) * Lq * 4;
  if ((Lq > 0 && (!dout || !dq || !lse)) || (Lk > 0 && (!dk || !dv))) return MHA_ERR_NULL;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                         reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) &
                        15u;
  if (mis || (reinterpret_cast<uintptr_t>(lse) & 3u)) return MHA_ERR_UNSUPPORTED;
  // gradients overlap nothing they are computed from, nor each other
  const void* ins[6] = {q, k, v, out, dout, lse};
  const size_t ins_b[6] = {qb, kb, kb, qb, qb, lb};
  void* outs[3] = {dq, dk, dv};
  const size_t outs_b[3] = {qb, kb, kb};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 6; ++i)
      if (overlaps(outs[o], outs_b[o], ins[i], ins_b[i])) return MHA_ERR_ALIAS;
    for (int o2 = o + 1; o2 < 3; ++o2)
      if (overlaps(outs[o], outs_b[o], outs[o2], outs_b[o2])) return MHA_ERR_ALIAS;
  }
  const size_t need = align256(lb);
  if (Lq > 0 && Lk > 0 && (!workspace || workspace_bytes < need ||
                            (reinterpret_cast<uintptr_t>(workspace) & 15u)))
    return MHA_ERR_WORKSPACE;
  // the workspace (D_i, written by the first kernel) overlaps no argument
  if (Lq > 0 && Lk > 0) {
    for (int i = 0; i < 6; ++i)
      if (overlaps(workspace, need, ins[i], ins_b[i])) return MHA_ERR_ALIAS;
    for (int o = 0; o < 3; ++o)
      if (overlaps(workspace, need, outs[o], outs_b[o])) return MHA_ERR_ALIAS;
  }
  DeviceState* dev = nullptr;
  rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // no queries: no gradient reaches the keys; no keys: every row's output is 0
  if (Lq == 0 || Lk == 0) {
    if (Lq > 0 && cudaMemsetAsync(dq, 0, qb, s) != cudaSuccess) return MHA_ERR_LAUNCH;
    if (Lk > 0 && (cudaMemsetAsync(dk, 0, kb, s) != cudaSuccess ||
                   cudaMemsetAsync(dv, 0, kb, s) != cudaSuccess))
      return MHA_ERR_LAUNCH;
    return MHA_OK;
  }
  if (bh * ((Lk + 127) / 128) > 0x7fffffffll || bh * ((Lq + 127) / 128) > 0x7fffffffll)
    return MHA_ERR_SHAPE;
  mha::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_map(&p.tm_q, q, B, Lq, H, d_k) || !encode_map(&p.tm_k, k, B, Lk, H, d_k) ||
      !encode_map(&p.tm_v, v, B, Lk, H, d_k) || !encode_map(&p.tm_do, dout, B, Lq, H, d_k) ||
      !encode_map(&p.tm_o, out, B, Lq, H, d_k) || !encode_map(&p.tm_dk, dk, B, Lk, H, d_k) ||
      !encode_map(&p.tm_dv, dv, B, Lk, H, d_k))
    return MHA_ERR_UNSUPPORTED;
  p.out = out;
  p.dout = dout;
  p.lse = lse;
  p.dvec = static_cast<float*>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.key_lens = key_lens;
  p.status = dev->status;
  p.B = B;
  p.H = H;
  p.Lq = Lq;
  p.Lk = Lk;
  p.mask_kind = mask_kind;
  p.d = d_k;
  p.scale = effective_scale(scale, d_k);
  p.scale_log2 = p.scale * kLog2e;
  return mha::launch_bwd(p, bf16_kernel_width(d_k, d_k), s, &t_info) == cudaSuccess
             ? MHA_OK
             : MHA_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// The multi-head layer: projections (the tcgen05 GEMM) around the attention
// kernel.
// ---------------------------------------------------------------------------
// 2-D map over a row-major bf16 matrix [rows, cols] with `ld` elements
// between rows; box = box_cols x box_rows, 128-byte swizzle (box_cols 64).
static bool encode_2d(CUtensorMap* m, const void* base, long long rows, long long cols,
                      long long ld, int box_cols, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// C[M x N] = A[M x K] B[K x N] (row-major bf16, leading dimensions in
// elements: multiples of 8, bases 16-byte aligned) on the tensor cores.
static int gemm_bf16(int M, int N, int K, const void* A, long long lda, const void* B,
                     long long ldb, void* C, long long ldc, DeviceState* dev, cudaStream_t s,
                     mha::LaunchInfo* info) {
  mha::GemmParams p;
  std::memset(&p, 0, sizeof(p));
  // (A is loaded in 128-row boxes: a 256-row tile takes two)
  if (!encode_2d(&p.tm_a, A, M, K, lda, 64, 128) || !encode_2d(&p.tm_b, B, K, N, ldb, 64, 64) ||
      !encode_2d(&p.tm_c, C, M, N, ldc, 64, 32))
    return MHA_ERR_UNSUPPORTED;
  p.status = dev->status;
  p.M = M;
  p.N = N;
  p.K = K;
  return mha::launch_gemm(p, s, info) == cudaSuccess ? MHA_OK : MHA_ERR_LAUNCH;
}

// workspace: [Q|K|V projections][O (heads concatenated)]
static size_t layer_proj_bytes(int B, int Lq, int Lk, size_t hd) {
  return align256((static_cast<size_t>(B) * Lq * hd + static_cast<size_t>(B) * Lk * 2 * hd) * 2);
}

size_t mha_layer_workspace_bytes(int B, int Lq, int Lk, int d_model, int H, int d_k) {
  if (B < 0 || Lq < 0 || Lk < 0 || d_model < 1 || H < 1 || !bf16_width_ok(d_k)) return 0;
  const size_t hd = static_cast<size_t>(H) * d_k;
  return layer_proj_bytes(B, Lq, Lk, hd) + align256(static_cast<size_t>(B) * Lq * hd * 2);
}

int mha_gemm_bf16(const void* a, const void* b, void* c, int M, int N, int K, long long lda,
                  long long ldb, long long ldc, void* stream) {
  t_info = mha::LaunchInfo{};
  if (M < 0 || N < 0 || K < 0) return MHA_ERR_SHAPE;
  if (M == 0 || N == 0) return MHA_OK;
  // (with K == 0 only c is touched: a and b may be NULL, their strides unused)
  if (!c || (K > 0 && (!a || !b))) return MHA_ERR_NULL;
  if (ldc < N || ldc > (1ll << 40) ||
      (K > 0 && (lda < K || ldb < N || lda > (1ll << 40) || ldb > (1ll << 40))))
    return MHA_ERR_SHAPE;
  if (ldc % 8 != 0 || (reinterpret_cast<uintptr_t>(c) & 15u) ||
      (K > 0 && ((lda | ldb) % 8 != 0 ||
                 ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u))))
    return MHA_ERR_UNSUPPORTED;
  const size_t cb = (static_cast<size_t>(M - 1) * ldc + N) * 2;
  if (K > 0 && (overlaps(c, cb, a, (static_cast<size_t>(M - 1) * lda + K) * 2) ||
                overlaps(c, cb, b, (static_cast<size_t>(K - 1) * ldb + N) * 2)))
    return MHA_ERR_ALIAS;
  DeviceState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {  // an empty sum: C = 0, row by row
    if (cudaMemset2DAsync(c, static_cast<size_t>(ldc) * 2, 0, static_cast<size_t>(N) * 2, M, s) !=
        cudaSuccess)
      return MHA_ERR_LAUNCH;
    return MHA_OK;
  }
  return gemm_bf16(M, N, K, a, lda, b, ldb, c, ldc, dev, s, &t_info);
}

int mha_layer_fwd(const void* x, const void* mem, const void* w_qkv, const void* w_o, void* y,
                  int B, int Lq, int Lk, int d_model, int H, int d_k, int mask_kind,
                  const int32_t* key_lens, float scale, void* workspace, size_t workspace_bytes,
                  void* stream) {
  t_info = mha::LaunchInfo{};
  if (B < 0 || Lq < 0 || Lk < 0 || d_model < 1 || H < 1 || d_k < 1) return MHA_ERR_SHAPE;
  if (!mask_known(mask_kind)) return MHA_ERR_MASK;
  if (has_causal(mask_kind) && Lq != Lk) return MHA_ERR_SHAPE;
  if (!mem && Lk != Lq) return MHA_ERR_SHAPE;  // self-attention: keys are the query rows
  if (!std::isfinite(scale) || scale < 0.f) return MHA_ERR_SCALE;
  if (!bf16_width_ok(d_k) || d_model % 8 != 0) return MHA_ERR_UNSUPPORTED;
  const long long hd = static_cast<long long>(H) * d_k;
  const long long rows_q = static_cast<long long>(B) * Lq, rows_k = static_cast<long long>(B) * Lk;
  if (rows_q > 0x7fffffffll || rows_k > 0x7fffffffll || hd * 3 > 0x7fffffffll ||
      (rows_q + rows_k) * (3 * hd + d_model) > (1ll << 40))
    return MHA_ERR_SHAPE;
  if (rows_q == 0) return MHA_OK;
  if (!x || !w_qkv || !w_o || !y) return MHA_ERR_NULL;
  if (has_padding(mask_kind) && !key_lens) return MHA_ERR_MASK;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(mem) |
       reinterpret_cast<uintptr_t>(w_qkv) | reinterpret_cast<uintptr_t>(w_o) |
       reinterpret_cast<uintptr_t>(y)) & 15u)
    return MHA_ERR_UNSUPPORTED;
  const size_t need = mha_layer_workspace_bytes(B, Lq, Lk, d_model, H, d_k);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MHA_ERR_WORKSPACE;
  const size_t xb = static_cast<size_t>(rows_q) * d_model * 2;
  const size_t mb = mem ? static_cast<size_t>(rows_k) * d_model * 2 : 0;
  const size_t wqb = static_cast<size_t>(d_model) * 3 * hd * 2, wob = static_cast<size_t>(hd) * d_model * 2;
  const void* ins[4] = {x, mem, w_qkv, w_o};
  const size_t ins_b[4] = {xb, mb, wqb, wob};
  for (int i = 0; i < 4; ++i)
    if (overlaps(y, xb, ins[i], ins_b[i]) || overlaps(workspace, need, ins[i], ins_b[i]))
      return MHA_ERR_ALIAS;
  if (overlaps(y, xb, workspace, need)) return MHA_ERR_ALIAS;
  DeviceState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Lk == 0) {  // every head's output is 0, and so is its projection
    return cudaMemsetAsync(y, 0, xb, s) == cudaSuccess ? MHA_OK : MHA_ERR_LAUNCH;
  }
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint16_t* proj = reinterpret_cast<uint16_t*>(w);
  uint16_t* o = reinterpret_cast<uint16_t*>(w + layer_proj_bytes(B, Lq, Lk, hd));
  const uint16_t* wq = static_cast<const uint16_t*>(w_qkv);
  const void *q, *k, *v;
  long long q_row, kv_row;
  mha::LaunchInfo gemms;  // the projection launches (the attention's own info is kept apart)
  if (!mem) {
    // one GEMM: [Q | K | V] = x [W^Q | W^K | W^V], rows of 3 H d_k
    rc = gemm_bf16(static_cast<int>(rows_q), static_cast<int>(3 * hd), d_model, x, d_model,
                   w_qkv, 3 * hd, proj, 3 * hd, dev, s, &gemms);
    if (rc != MHA_OK) return rc;
    q = proj;
    k = proj + hd;
    v = proj + 2 * hd;
    q_row = kv_row = 3 * hd;
  } else {
    // Q = x W^Q (rows of H d_k) and [K | V] = mem [W^K | W^V] (rows of 2 H d_k),
    // reading the weight's column blocks in place (leading dimension 3 H d_k)
    uint16_t* kv = proj + rows_q * hd;
    rc = gemm_bf16(static_cast<int>(rows_q), static_cast<int>(hd), d_model, x, d_model, wq,
                   3 * hd, proj, hd, dev, s, &gemms);
    if (rc == MHA_OK)
      rc = gemm_bf16(static_cast<int>(rows_k), static_cast<int>(2 * hd), d_model, mem, d_model,
                     wq + hd, 3 * hd, kv, 2 * hd, dev, s, &gemms);
    if (rc != MHA_OK) return rc;
    q = proj;
    k = kv;
    v = kv + hd;
    q_row = hd;
    kv_row = 2 * hd;
  }
  // the heads' attention, read in place from the projections; O comes out as
  // [B, Lq, H, d_k] = the heads' concatenation, rows of H d_k
  rc = attention_bf16(q, k, v, o, nullptr, q_row, kv_row, kv_row, B, H, Lq, Lk, d_k, d_k,
                      mask_kind, key_lens, scale, dev, s);
  if (rc != MHA_OK) return rc;
  const mha::LaunchInfo attn = t_info;
  // y = Concat(heads) W^O
  rc = gemm_bf16(static_cast<int>(rows_q), d_model, static_cast<int>(hd), o, hd, w_o, d_model, y,
                 d_model, dev, s, &gemms);
  if (rc != MHA_OK) return rc;
  // every launch of the layer is this library's: the GEMMs and the attention
  t_info = attn;
  t_info.kernels = attn.kernels + gemms.kernels;
  return MHA_OK;
}

size_t mha_fwd_host_workspace_bytes(int B, int H, int Lq, int Lk, int d_k, int elem_bytes) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || d_k < 1) return 0;
  if (elem_bytes != 2 && elem_bytes != 4) return 0;
  const size_t qb = static_cast<size_t>(B) * Lq * H * d_k * elem_bytes;
  const size_t kb = static_cast<size_t>(B) * Lk * H * d_k * elem_bytes;
  return align256(qb) * 2 + align256(kb) * 2 + align256(static_cast<size_t>(B) * 4);
}

int mha_fwd_host(const void* q, const void* k, const void* v, void* out, int B, int H, int Lq,
                 int Lk, int d_k, int mask_kind, const int32_t* key_lens, float scale,
                 int elem_bytes, void* workspace, size_t workspace_bytes, void* stream) {
  if (elem_bytes != 2 && elem_bytes != 4) return MHA_ERR_UNSUPPORTED;
  const size_t need = mha_fwd_host_workspace_bytes(B, H, Lq, Lk, d_k, elem_bytes);
  if (need == 0) return MHA_ERR_SHAPE;
  const size_t qb = static_cast<size_t>(B) * Lq * H * d_k * elem_bytes;
  const size_t kb = static_cast<size_t>(B) * Lk * H * d_k * elem_bytes;
  if (qb == 0) return MHA_OK;
  if (!workspace || workspace_bytes < need) return MHA_ERR_WORKSPACE;
  if (!q || !out || (kb > 0 && (!k || !v))) return MHA_ERR_NULL;
  if (!mask_known(mask_kind)) return MHA_ERR_MASK;
  if (has_padding(mask_kind) && !key_lens) return MHA_ERR_MASK;
  HostPipe* pipe = nullptr;
  if (host_pipe(&pipe) != MHA_OK) return MHA_ERR_LAUNCH;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint8_t* dq = w;
  uint8_t* dk = dq + align256(qb);
  uint8_t* dv = dk + align256(kb);
  uint8_t* dout = dv + align256(kb);
  int32_t* dlens = reinterpret_cast<int32_t*>(dout + align256(qb));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t* lens = nullptr;
  if (has_padding(mask_kind)) {
    if (cudaMemcpyAsync(dlens, key_lens, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return MHA_ERR_LAUNCH;
    lens = dlens;
  }
  // Sequences are independent and each one's rows are contiguous in every
  // tensor, so the batch goes in chunks of sequences over two streams: the
  // copies in of one chunk, the kernel of the one before and the copy out of
  // the one before that overlap.  Both streams start after the work already
  // on the caller's stream, which waits for both at the end.  Chunks carry at
  // least 8 MiB of inputs: below that a chunk's own launch costs more than
  // the overlap saves (measured: 32 sequences of 128 rows, 12.6 MB, took
  // 168 us in four chunks against 128 us in one).
  const size_t in_bytes = qb + 2 * kb;
  long long chunks = static_cast<long long>(in_bytes >> 23);
  if (chunks > 4) chunks = 4;
  if (chunks > B) chunks = B;
  const int n_chunks = chunks < 1 ? 1 : static_cast<int>(chunks);
  const size_t q_seq = qb / B, k_seq = kb / B;
  std::unique_lock<std::mutex> queued(pipe->order);
  if (cudaEventRecord(pipe->start, s) != cudaSuccess ||
      cudaStreamWaitEvent(pipe->st[0], pipe->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(pipe->st[1], pipe->start, 0) != cudaSuccess)
    return MHA_ERR_LAUNCH;
  int rc = MHA_OK;
  for (int c = 0; c < n_chunks && rc == MHA_OK; ++c) {
    const int b0 = static_cast<int>(static_cast<long long>(B) * c / n_chunks);
    const int b1 = static_cast<int>(static_cast<long long>(B) * (c + 1) / n_chunks);
    const int nb = b1 - b0;
    cudaStream_t x = pipe->st[c & 1];
    const size_t qo = q_seq * b0, ko = k_seq * b0;
    if (cudaMemcpyAsync(dq + qo, static_cast<const uint8_t*>(q) + qo, q_seq * nb,
                        cudaMemcpyHostToDevice, x) != cudaSuccess ||
        (kb > 0 && (cudaMemcpyAsync(dk + ko, static_cast<const uint8_t*>(k) + ko, k_seq * nb,
                                    cudaMemcpyHostToDevice, x) != cudaSuccess ||
                    cudaMemcpyAsync(dv + ko, static_cast<const uint8_t*>(v) + ko, k_seq * nb,
                                    cudaMemcpyHostToDevice, x) != cudaSuccess))) {
      rc = MHA_ERR_LAUNCH;
      break;
    }
    rc = (elem_bytes == 2)
             ? mha_fwd(dq + qo, kb ? dk + ko : nullptr, kb ? dv + ko : nullptr, dout + qo, nb, H, Lq,
                       Lk, d_k, mask_kind, lens ? lens + b0 : nullptr, scale, x)
             : mha_fwd_f32(dq + qo, kb ? dk + ko : nullptr, kb ? dv + ko : nullptr, dout + qo, nb,
                           H, Lq, Lk, d_k, mask_kind, lens ? lens + b0 : nullptr, scale, x);
    if (rc != MHA_OK) break;
    if (cudaMemcpyAsync(static_cast<uint8_t*>(out) + qo, dout + qo, q_seq * nb,
                        cudaMemcpyDeviceToHost, x) != cudaSuccess)
      rc = MHA_ERR_LAUNCH;
  }
  for (int i = 0; i < 2; ++i) {
    if (cudaEventRecord(pipe->done[i], pipe->st[i]) != cudaSuccess ||
        cudaStreamWaitEvent(s, pipe->done[i], 0) != cudaSuccess)
      rc = rc == MHA_OK ? MHA_ERR_LAUNCH : rc;
  }
  queued.unlock();
  if (rc != MHA_OK) {
    cudaStreamSynchronize(s);
    return rc;
  }
  return mha_sync_status(stream);
}

int mha_selftest_timeout(void* stream) {
  t_info = mha::LaunchInfo{};
  DeviceState* dev = nullptr;
  const int rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status);
  t_info.kernels = 1;
  t_info.grid = 1;
  t_info.block = 32;
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_LAUNCH;
}

void mha_debug_withhold_p(int on) { g_withhold_p = on ? 1 : 0; }

int mha_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MHA_ERR_LAUNCH;
  DeviceState* dev = nullptr;
  const int rc = device_state(&dev);
  if (rc != MHA_OK) return rc;
  DeviceStatus st;
  if (cudaMemcpy(&st, dev->status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MHA_ERR_LAUNCH;
  if (st.code != 0) {
    const DeviceStatus zero = {0, 0, 0, 0};
    if (cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MHA_ERR_LAUNCH;
  }
  return st.code;
}

const char* mha_status_string(int status) {
  switch (status) {
    case MHA_OK: return "ok";
    case MHA_ERR_NULL: return "a required pointer is NULL";
    case MHA_ERR_SHAPE: return "bad sizes (negative, causal with Lq != Lk, or too large)";
    case MHA_ERR_UNSUPPORTED:
      return "unsupported (d_k for this dtype, pointer alignment, or device is not sm_103)";
    case MHA_ERR_MASK: return "unknown mask kind, or key_lens missing under key padding";
    case MHA_ERR_SCALE: return "scale must be finite and >= 0 (0 selects 1/sqrt(d_k))";
    case MHA_ERR_LAUNCH: return "a CUDA call failed";
    case MHA_ERR_TIMEOUT: return "a pipeline wait on the device timed out";
    case MHA_ERR_ALIAS: return "out (or lse) overlaps q, k or v (or out)";
    case MHA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

void mha_last_launch_info(int* kernels, int* grid, int* block, int* smem_bytes) {
  if (kernels) *kernels = t_info.kernels;
  if (grid) *grid = t_info.grid;
  if (block) *block = t_info.block;
  if (smem_bytes) *smem_bytes = t_info.smem;
}

}  // extern "C"
