// mha_gemm.cu -- the projection GEMMs of the multi-head layer on the
// 5th-generation tensor cores (TMA + tcgen05 + TMEM), sm_103a.
//
// Row-major C[M x N] = A[M x K] B[K x N], bf16 operands, float32
// accumulation, bf16 result: the products x W^Q, m W^K, m W^V and
// Concat(head_1..head_H) W^O of "Attention Is All You Need", Section 3.2.2.
//
// Tiles of 128 x 256 outputs, K in blocks of 64.  Persistent CTAs (one per
// SM) walk the tiles in groups of 16 row blocks, so the A row panels and B
// column panels of the tiles running at once stay in L2.  Six warps:
//   warp 0     TMA producer: the A block (128 rows x 64 k, K-major) and four
//              B blocks (64 k x 64 n, N-major) of each k step into a 4-stage
//              ring (48 KB a stage)
//   warp 1     TMEM allocator and MMA issuer: tcgen05.mma kind::f16 M128
//              N256 K16, four per k step, into one of two 256-column float32
//              accumulators, so a tile's epilogue overlaps the next tile's
//              products
//   warps 2-5  epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its 32
//              output rows), rounds to bf16, stages 64 columns at a time in
//              shared memory (128-byte swizzle) and writes them with a TMA
//              store; each warp stages and stores its own rows, so the
//              epilogue needs no barrier across warps
// With a long K (a tile's products take far longer than its epilogue) the
// tiles are 256 x 256 instead: two 128-row accumulators (all 512 TMEM
// columns) share every B block, so each k step moves 64 KB through TMA for
// 1024 tensor cycles instead of 48 KB for 512 -- two thirds of the L2 to
// shared-memory traffic per flop -- at the cost of the epilogue no longer
// overlapping the next tile (one accumulator pair, three 64 KB stages).
// Rows, columns and k past the matrix edges are read as zero by the tensor
// maps and never written.  Every wait is bounded: a role that gives up
// raises the CTA's abort flag, the others follow, each waits for its own
// copies and tensor-core work, and the status word records MHA_ERR_TIMEOUT.
#include <cuda_bf16.h>

#include "kernels.h"

namespace mha {
namespace {

constexpr int kGemmThreads = 192;
constexpr int kGemmBN = 256, kGemmBK = 64;
constexpr int kGemmProducerWarp = 0, kGemmMmaWarp = 1;
constexpr int kRoleGemmProducer = 8, kRoleGemmMma = 9, kRoleGemmEpilogue = 10;

// TALL: 256-row tiles (two 128-row accumulators, no second accumulator set);
// otherwise 128-row tiles with two accumulators in turn.
template <bool TALL>
struct GemmCfg {
  static constexpr int BM = TALL ? 256 : 128;
  static constexpr int HALVES = BM / 128;                        // 128-row accumulators per tile
  static constexpr int ACC_SETS = TALL ? 1 : 2;                  // tiles in TMEM at once
  static constexpr int STAGES = TALL ? 3 : 4;
  static constexpr int GROUP_M = TALL ? 8 : 16;                  // row blocks walked together (L2 reuse)
  static constexpr int A_HALF = 128 * kGemmBK * 2;               // 128 rows x 128 B
  static constexpr int A_BYTES = HALVES * A_HALF;
  static constexpr int B_CHUNK = kGemmBK * 128;                  // 64 k rows x 64 n (128 B)
  static constexpr int B_BYTES = (kGemmBN / 64) * B_CHUNK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;          // 48 KB, or 64 KB when TALL
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OUT_CHUNK = 32 * 128;                     // one warp's 32 rows x 64 bf16
  static constexpr int OFF_OUT = OFF_B + STAGES * B_BYTES;       // 4 warps x 2 buffers
  static constexpr int OFF_BAR = OFF_OUT + 8 * OUT_CHUNK;
  static constexpr int FULL = 0, EMPTY = STAGES, ACC_FULL = 2 * STAGES,
                       ACC_EMPTY = 2 * STAGES + 2, DRAIN = 2 * STAGES + 4;
  static constexpr int NBAR = 2 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;            // TMEM slot, abort flag
  static constexpr int SMEM = OFF_MISC + 16 + 1024;              // + slack to align to 1024
  static constexpr uint32_t TMEM_COLS = 512;                     // 2 x 256 float32 columns
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(OFF_B % 1024 == 0 && OFF_OUT % 1024 == 0 && OFF_BAR % 8 == 0, "alignment");
};

// Output tile t: groups of GROUP_M row blocks, row block fastest inside a
// group, so the tiles that run at once share A row panels and B column panels.
template <bool TALL>
__device__ __forceinline__ void gemm_tile(const GemmParams& p, int t, int& m0, int& n0) {
  constexpr int G = GemmCfg<TALL>::GROUP_M;
  const int per_group = G * p.tiles_n;
  const int group = t / per_group;
  const int first = group * G;
  const int rows = min(G, p.tiles_m - first);
  const int in = t - group * per_group;
  m0 = (first + in % rows) * GemmCfg<TALL>::BM;
  n0 = (in / rows) * kGemmBN;
}

template <bool TALL>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<TALL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sA = s_base + C::OFF_A, sB = s_base + C::OFF_B, sOut = s_base + C::OFF_OUT;
  auto bar = [&](int id) { return s_base + C::OFF_BAR + 8u * static_cast<uint32_t>(id); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int n_tiles = p.tiles_m * p.tiles_n;
  constexpr int S = C::STAGES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(C::FULL + s), 1);
      mbar_init(bar(C::EMPTY + s), 1);
    }
    for (int a = 0; a < C::ACC_SETS; ++a) {
      mbar_init(bar(C::ACC_FULL + a), 1);
      mbar_init(bar(C::ACC_EMPTY + a), 128);
    }
    mbar_init(bar(C::DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kGemmProducerWarp && lane == 0) {
    tma_prefetch_desc(&p.tm_a);
    tma_prefetch_desc(&p.tm_b);
    tma_prefetch_desc(&p.tm_c);
  }
  if (warp == kGemmMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // no global memory before this point: the set-up may overlap the previous
  // kernel on the stream
  griddep_wait();

  if (warp == kGemmProducerWarp) {
    // ---- TMA producer: k step g of the CTA goes to stage g % S
    const int site = kRoleGemmProducer * 64;
    int g = 0;
    bool ok = true;
    for (int t = static_cast<int>(blockIdx.x); ok && t < n_tiles; t += static_cast<int>(gridDim.x)) {
      int m0, n0;
      gemm_tile<TALL>(p, t, m0, n0);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const int s = g % S;
        if (g >= S && !mbar_wait(bar(C::EMPTY + s), ((g / S) - 1) & 1, abort_flag, p.status,
                                 site + C::EMPTY + s)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::FULL + s), C::STAGE_BYTES);
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            tma_load_2d(sA + s * C::A_BYTES + hf * C::A_HALF, &p.tm_a, bar(C::FULL + s),
                        kb * kGemmBK, m0 + 128 * hf);
#pragma unroll
          for (int j = 0; j < kGemmBN / 64; ++j)
            tma_load_2d(sB + s * C::B_BYTES + j * C::B_CHUNK, &p.tm_b, bar(C::FULL + s),
                        n0 + 64 * j, kb * kGemmBK);
        }
        __syncwarp();
        ++g;
      }
    }
    // every copy this warp started must land before the CTA exits (waits that
    // ignore the abort flag; the normal path finds them complete)
    volatile int never = 0;
    for (int i = (g > S ? g - S : 0); i < g; ++i)
      mbar_wait(bar(C::FULL + i % S), (i / S) & 1, &never, p.status, site + C::FULL);
  } else if (warp == kGemmMmaWarp) {
    // ---- MMA issuer: A K-major (8-row groups 1024 B apart, +32 B per K16
    // step inside the 128-byte swizzle atom); B N-major (64-wide n chunks
    // B_CHUNK apart, 8-row k groups 1024 B apart, +2048 B per K16 step)
    const int site = kRoleGemmMma * 64;
    constexpr uint32_t idesc = idesc_bf16_f32(128, kGemmBN, false, true);
    const uint64_t da0 = smem_desc_sw128(sA, 16, 1024);
    const uint64_t db0 = smem_desc_sw128(sB, C::B_CHUNK, 1024);
    int g = 0, i = 0;
    bool ok = true;
    for (int t = static_cast<int>(blockIdx.x); ok && t < n_tiles;
         t += static_cast<int>(gridDim.x), ++i) {
      const int a = C::ACC_SETS == 2 ? (i & 1) : 0;
      const int use = C::ACC_SETS == 2 ? (i >> 1) : i;  // earlier tiles in this accumulator set
      // the epilogue must have read this accumulator set's previous tile
      if (use >= 1 && !mbar_wait(bar(C::ACC_EMPTY + a), (use - 1) & 1, abort_flag, p.status,
                                 site + C::ACC_EMPTY + a)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + static_cast<uint32_t>(a * kGemmBN);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const int s = g % S;
        if (!mbar_wait(bar(C::FULL + s), (g / S) & 1, abort_flag, p.status, site + C::FULL + s)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t da = da0 + static_cast<uint64_t>((s * C::A_BYTES) >> 4);
          const uint64_t db = db0 + static_cast<uint64_t>((s * C::B_BYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < kGemmBK / 16; ++ks)
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
              umma_ss(acc + static_cast<uint32_t>(hf * kGemmBN),
                      da + static_cast<uint64_t>((hf * C::A_HALF + ks * 32) >> 4),
                      db + static_cast<uint64_t>((ks * 2048) >> 4), idesc, (kb | ks) ? 1u : 0u);
          umma_commit(bar(C::EMPTY + s));  // the stage is free once these are done
        }
        __syncwarp();
        ++g;
      }
      if (!ok) break;
      if (elect_one()) umma_commit(bar(C::ACC_FULL + a));
      __syncwarp();
    }
    // every MMA this warp issued completes before TMEM is released
    if (elect_one()) umma_commit(bar(C::DRAIN));
    __syncwarp();
    volatile int never = 0;
    mbar_wait(bar(C::DRAIN), 0, &never, p.status, site + C::DRAIN);
  } else {
    // ---- epilogue: warp w's 32 rows of each tile, 64 columns at a time
    const int site = kRoleGemmEpilogue * 64;
    const int q = warp & 3;                      // TMEM lane quarter
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t out_base = sOut + static_cast<uint32_t>(q * 2 * C::OUT_CHUNK);
    int i = 0, chunks = 0;
    bool prev_stored = true;  // the previous chunk issued a TMA store
    for (int t = static_cast<int>(blockIdx.x); t < n_tiles; t += static_cast<int>(gridDim.x), ++i) {
      const int a = C::ACC_SETS == 2 ? (i & 1) : 0;
      const int use = C::ACC_SETS == 2 ? (i >> 1) : i;
      if (!mbar_wait(bar(C::ACC_FULL + a), use & 1, abort_flag, p.status, site + C::ACC_FULL + a))
        break;
      tc_fence_after();
      int m0, n0;
      gemm_tile<TALL>(p, t, m0, n0);
      // chunk cc: accumulator half cc / 4 (rows 128 (cc / 4) ..), columns 64 (cc % 4) ..
#pragma unroll 1
      for (int cc = 0; cc < C::HALVES * (kGemmBN / 64); ++cc, ++chunks) {
        const int hf = cc / (kGemmBN / 64), c = cc % (kGemmBN / 64);
        const uint32_t tacc = tmem + lane_off + static_cast<uint32_t>((a + hf) * kGemmBN);
        uint32_t r[64];
        tmem_ld32(tacc + 64u * c, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(tacc + 64u * c + 32u, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
        if (cc == C::HALVES * (kGemmBN / 64) - 1) {
          // the accumulator may take the next tile from here on
          tc_fence_before();
          mbar_arrive(bar(C::ACC_EMPTY + a));
        }
        const uint32_t stage = out_base + static_cast<uint32_t>((chunks & 1) * C::OUT_CHUNK);
        // The store issued from this buffer two chunks ago must have read it:
        // with the previous chunk's store committed after it, at most one
        // group may still be reading; when the previous chunk stored nothing
        // (its box lay wholly past the matrix), none may.
        if (lane == 0) {
          if (prev_stored) {
            tma_store_wait_read_1();
          } else {
            tma_store_wait_read();
          }
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r[8 * u + 2 * e]), __uint_as_float(r[8 * u + 2 * e + 1]));
          st_shared_v4(stage + static_cast<uint32_t>(lane * 128) +
                           (static_cast<uint32_t>(u ^ (lane & 7)) << 4),
                       w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        // (a box wholly past the matrix's last row or column is not stored)
        const int row0 = m0 + 128 * hf + 32 * q;
        prev_stored = n0 + 64 * c < p.N && row0 < p.M;
        if (lane == 0 && prev_stored) {
          tma_store_2d(&p.tm_c, stage, n0 + 64 * c, row0);
          tma_store_commit();
        }
        __syncwarp();
      }
    }
    // the staging buffers must outlive the reads of the last stores, and the
    // writes must be complete before the grid ends
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kGemmMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

namespace {

template <bool TALL>
cudaError_t launch_gemm_t(const GemmParams& params, cudaStream_t stream, LaunchInfo* info) {
  using C = GemmCfg<TALL>;
  GemmParams p = params;
  p.tiles_m = (p.M + C::BM - 1) / C::BM;
  p.tiles_n = (p.N + kGemmBN - 1) / kGemmBN;
  p.k_blocks = (p.K + kGemmBK - 1) / kGemmBK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  static int sms[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(gemm_bf16_kernel<TALL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (tiles <= 0 || tiles > 0x7fffffffll) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(tiles < sms[dev] ? tiles : sms[dev]);
  e = launch_serialized(gemm_bf16_kernel<TALL>, dim3(grid), dim3(kGemmThreads), C::SMEM, stream, p);
  if (e != cudaSuccess) return e;
  if (info) {
    info->kernels += 1;
    info->grid = grid;
    info->block = kGemmThreads;
    info->smem = C::SMEM;
  }
  return cudaGetLastError();
}

}  // namespace

// The 256-row tiles when K is long enough that a tile's products (K / 64 k
// steps of 1024 tensor cycles) dwarf its epilogue, which they do not overlap
// (measured: +9 to +12 % at K 4096 to 12288 against the 128-row tiles, -5 %
// at K 512).
constexpr int kGemmTallMinK = 4096;

cudaError_t launch_gemm(const GemmParams& p, cudaStream_t stream, LaunchInfo* info) {
  return p.K >= kGemmTallMinK ? launch_gemm_t<true>(p, stream, info)
                              : launch_gemm_t<false>(p, stream, info);
}

}  // namespace mha
