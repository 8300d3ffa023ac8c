// mha_gemm.cu -- the plain projection GEMMs of the multi-head layer, on
// cuBLASLt (a library GEMM: bf16 operands, float32 accumulation, bf16 result).
//
// Row-major C[M x N] = A[M x K] B[K x N] with leading dimensions (elements
// between consecutive rows) lda, ldb, ldc.  cuBLASLt is column-major, where a
// row-major matrix is its own transpose, so the call computes
//   C^T (N x M, ld ldc) = B^T (N x K, ld ldb) A^T (K x M, ld lda)
// with no transposed copies.  One cuBLASLt handle per device, created on
// first use.
#include <cublasLt.h>

#include <mutex>

#include "kernels.h"

namespace mha {
namespace {

cublasLtHandle_t g_lt[64] = {};
std::mutex g_lt_mutex;

cublasLtHandle_t lt_handle() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_lt_mutex);
  if (!g_lt[dev] && cublasLtCreate(&g_lt[dev]) != CUBLAS_STATUS_SUCCESS) g_lt[dev] = nullptr;
  return g_lt[dev];
}

// Owns the descriptors of one call.
struct LtCall {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  ~LtCall() {
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (c) cublasLtMatrixLayoutDestroy(c);
    if (b) cublasLtMatrixLayoutDestroy(b);
    if (a) cublasLtMatrixLayoutDestroy(a);
    if (op) cublasLtMatmulDescDestroy(op);
  }
};

}  // namespace

bool gemm_bf16_rowmajor(int M, int N, int K, const void* A, long long lda, const void* B,
                        long long ldb, void* C, long long ldc, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return true;
  cublasLtHandle_t h = lt_handle();
  if (!h) return false;
  LtCall call;
  if (cublasLtMatmulDescCreate(&call.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS)
    return false;
  // column-major operands: first = B^T (N x K), second = A^T (K x M), result C^T (N x M)
  if (cublasLtMatrixLayoutCreate(&call.a, CUDA_R_16BF, N, K, ldb) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&call.b, CUDA_R_16BF, K, M, lda) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&call.c, CUDA_R_16BF, N, M, ldc) != CUBLAS_STATUS_SUCCESS)
    return false;
  if (cublasLtMatmulPreferenceCreate(&call.pref) != CUBLAS_STATUS_SUCCESS) return false;
  const uint64_t ws = workspace ? workspace_bytes : 0;
  if (cublasLtMatmulPreferenceSetAttribute(call.pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                           &ws, sizeof(ws)) != CUBLAS_STATUS_SUCCESS)
    return false;
  cublasLtMatmulHeuristicResult_t heur = {};
  int found = 0;
  if (cublasLtMatmulAlgoGetHeuristic(h, call.op, call.a, call.b, call.c, call.c, call.pref, 1,
                                     &heur, &found) != CUBLAS_STATUS_SUCCESS ||
      found < 1)
    return false;
  const float alpha = 1.f, beta = 0.f;
  return cublasLtMatmul(h, call.op, &alpha, B, call.a, A, call.b, &beta, C, call.c, C, call.c,
                        &heur.algo, workspace, ws, stream) == CUBLAS_STATUS_SUCCESS;
}

}  // namespace mha
