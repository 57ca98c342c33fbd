// gemm.cpp -- cuBLASLt bf16 GEMMs for the layer's projections.
//
// Row-major C = A W^T is the column-major product C^T = W A^T: cuBLASLt sees
// W as a column-major K x N matrix taken transposed and A as a column-major
// K x M matrix, giving the column-major N x M matrix that is C row-major.
// One process-wide handle, created on first use; the algorithm chosen by
// cuBLASLt's heuristic is cached per problem shape.
#include "gemm.h"

#include <cublasLt.h>

#include <map>
#include <mutex>
#include <tuple>

namespace mamba {
namespace {

cublasLtHandle_t handle() {
  static cublasLtHandle_t h = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    if (cublasLtCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
  });
  return h;
}

using Key = std::tuple<long, int, int, int, int, bool, size_t>;

struct Plan {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
  cublasLtMatmulAlgo_t algo;
  bool ok = false;
};

std::mutex g_mu;
std::map<Key, Plan> g_plans;

Plan make_plan(long M, int N, int K, int lda, int ldc, bool bias, size_t ws_bytes) {
  Plan p;
  if (!handle()) return p;
  if (cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return p;
  const cublasOperation_t tA = CUBLAS_OP_T, tB = CUBLAS_OP_N;
  cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSA, &tA, sizeof(tA));
  cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSB, &tB, sizeof(tB));
  if (bias) {
    const cublasLtEpilogue_t ep = CUBLASLT_EPILOGUE_BIAS;
    cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_EPILOGUE, &ep, sizeof(ep));
  }
  // operand "A" of cuBLASLt: W as column-major K x N; "B": A as column-major K x M
  if (cublasLtMatrixLayoutCreate(&p.a, CUDA_R_16BF, K, N, K) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&p.b, CUDA_R_16BF, K, M, lda) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&p.c, CUDA_R_16BF, N, M, ldc) != CUBLAS_STATUS_SUCCESS)
    return p;
  cublasLtMatmulPreference_t pref = nullptr;
  if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) return p;
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof(ws_bytes));
  cublasLtMatmulHeuristicResult_t res;
  int found = 0;
  if (cublasLtMatmulAlgoGetHeuristic(handle(), p.op, p.a, p.b, p.c, p.c, pref, 1, &res, &found) ==
          CUBLAS_STATUS_SUCCESS &&
      found > 0) {
    p.algo = res.algo;
    p.ok = true;
  }
  cublasLtMatmulPreferenceDestroy(pref);
  return p;
}

}  // namespace

bool gemm_bf16(const void* A, int lda, const void* W, const void* bias, void* C, int ldc, long M, int N, int K,
               void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return M >= 0 && N >= 0;
  // the lock also covers the launch: the cached descriptor's bias pointer is
  // set per call
  std::lock_guard<std::mutex> lk(g_mu);
  const Key key{M, N, K, lda, ldc, bias != nullptr, ws_bytes};
  auto it = g_plans.find(key);
  if (it == g_plans.end()) it = g_plans.emplace(key, make_plan(M, N, K, lda, ldc, bias != nullptr, ws_bytes)).first;
  const Plan& p = it->second;
  if (!p.ok) return false;
  if (bias &&
      cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias)) !=
          CUBLAS_STATUS_SUCCESS)
    return false;
  const float one = 1.0f, zero = 0.0f;
  return cublasLtMatmul(handle(), p.op, &one, W, p.a, A, p.b, &zero, C, p.c, C, p.c, &p.algo, ws, ws_bytes,
                        stream) == CUBLAS_STATUS_SUCCESS;
}

}  // namespace mamba
