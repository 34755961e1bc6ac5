// linear.cu -- the projections around attention, as plain bf16 GEMMs on cuBLASLt.
//
// "Parallel multi-head attention", sections 2.1-2.3 and 3.1: the query, key and value
// projections are ColumnParallelLinear layers (each device holds the output columns of
// its heads), the output projection a RowParallelLinear (each device holds the input
// rows of its heads and the partial results are summed).  On one GPU the full weights
// are local and both are ordinary nn.Linear products, y = x W^T with W [out][in]:
//     forward   y[M][out]  = x[M][in] . W^T
//     backward  dx[M][in]  = dy[M][out] . W
//               dW[out][in] (+)= dy^T . x
// bf16 operands and results, fp32 accumulation.  These are plain library GEMMs, so they
// go to cuBLASLt (row-major matrices are handed over as their column-major transposes);
// no workspace is passed, so nothing is allocated on the device.
#include <cublasLt.h>

#include <mutex>

#include "internal.h"

namespace sp {
namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mutex;
cublasLtHandle_t g_handle[kMaxDevices] = {};

cublasLtHandle_t handle_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_handle[dev] == nullptr && cublasLtCreate(&g_handle[dev]) != CUBLAS_STATUS_SUCCESS)
    g_handle[dev] = nullptr;
  return g_handle[dev];
}

// Column-major GEMM  C[m][n] (ld = ldc) = op(A) op(B) (+ beta C), bf16, fp32 accumulation.
bool gemm_cm(bool trans_a, bool trans_b, int m, int n, int k, const void* a, int64_t lda,
             const void* b, int64_t ldb, void* c, int64_t ldc, float beta, cudaStream_t stream) {
  cublasLtHandle_t h = handle_for_current_device();
  if (h == nullptr) return false;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  bool ok = cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS;
  const cublasOperation_t ta = trans_a ? CUBLAS_OP_T : CUBLAS_OP_N;
  const cublasOperation_t tb = trans_b ? CUBLAS_OP_T : CUBLAS_OP_N;
  ok = ok && cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta) ==
                 CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb) ==
                 CUBLAS_STATUS_SUCCESS;
  // stored shapes (rows x cols, column-major) of A and B before op()
  ok = ok && cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, trans_a ? k : m, trans_a ? m : k, lda) ==
                 CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, trans_b ? n : k, trans_b ? k : n, ldb) ==
                 CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, m, n, ldc) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatmulPreferenceCreate(&pref) == CUBLAS_STATUS_SUCCESS;
  const size_t no_workspace = 0;
  ok = ok && cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                                  &no_workspace, sizeof no_workspace) ==
                 CUBLAS_STATUS_SUCCESS;
  cublasLtMatmulHeuristicResult_t heur;
  int found = 0;
  ok = ok && cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, lc, lc, pref, 1, &heur, &found) ==
                 CUBLAS_STATUS_SUCCESS &&
       found > 0;
  const float alpha = 1.0f;
  ok = ok && cublasLtMatmul(h, op, &alpha, a, la, b, lb, &beta, c, lc, c, lc, &heur.algo,
                            nullptr, 0, stream) == CUBLAS_STATUS_SUCCESS;
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return ok;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sp_status check_linear(int M, int in, int out) {
  if (M < 0 || in < 1 || out < 1) return SP_ERR_INVALID_ARG;
  if (in % 8 != 0 || out % 8 != 0) return SP_ERR_MISALIGNED;   // 16-byte rows
  return SP_OK;
}

}  // namespace
}  // namespace sp

using namespace sp;

extern "C" {

sp_status sp_linear_fwd(const void* x, const void* w, void* y, int M, int in, int out,
                        void* stream) {
  const sp_status st = check_linear(M, in, out);
  if (st != SP_OK) return st;
  if (x == nullptr || w == nullptr || y == nullptr) return SP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return SP_ERR_MISALIGNED;
  if (M == 0) return SP_OK;
  // y^T (out x M) = W (out x in) . x^T (in x M); W is stored column-major as in x out
  return gemm_cm(true, false, out, M, in, w, in, x, in, y, out, 0.0f,
                 static_cast<cudaStream_t>(stream))
             ? SP_OK
             : SP_ERR_CUDA;
}

sp_status sp_linear_bwd(const void* dy, const void* x, const void* w, void* dx, void* dw, int M,
                        int in, int out, int accumulate_dw, void* stream) {
  const sp_status st = check_linear(M, in, out);
  if (st != SP_OK) return st;
  if (dy == nullptr || x == nullptr || w == nullptr || (dx == nullptr && dw == nullptr))
    return SP_ERR_INVALID_ARG;
  if (accumulate_dw != 0 && accumulate_dw != 1) return SP_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(w) || (dx && !aligned16(dx)) ||
      (dw && !aligned16(dw)))
    return SP_ERR_MISALIGNED;
  if (M == 0) return SP_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // dx^T (in x M) = W^T (in x out) . dy^T (out x M)
  if (dx != nullptr && !gemm_cm(false, false, in, M, out, w, in, dy, out, dx, in, 0.0f, s))
    return SP_ERR_CUDA;
  // dW^T (in x out) = x^T (in x M) . dy (M x out)
  if (dw != nullptr &&
      !gemm_cm(false, true, in, out, M, x, in, dy, out, dw, in, accumulate_dw ? 1.0f : 0.0f, s))
    return SP_ERR_CUDA;
  return SP_OK;
}

}  // extern "C"
