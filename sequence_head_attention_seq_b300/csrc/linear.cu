// linear.cu -- the projections around attention, on the library's tcgen05 GEMM.
//
// "Parallel multi-head attention", sections 2.1-2.3 and 3.1: the query, key and value
// projections are ColumnParallelLinear layers (each device holds the output columns of
// its heads), the output projection a RowParallelLinear (each device holds the input
// rows of its heads and the partial results are summed).  On one GPU the full weights
// are local and both are ordinary nn.Linear products, y = x W^T with W [out][in]:
//     forward   y[M][out]  = x[M][in] . W^T        A = x (K-major),  B = W (K-major)
//     backward  dx[M][in]  = dy[M][out] . W        A = dy (K-major), B = W (MN-major)
//               dW[out][in] (+)= dy^T . x          A = dy (MN-major), B = x (MN-major)
// bf16 operands and results, fp32 accumulation (gemm.cu); nothing is allocated.
#include "internal.h"

namespace sp {
namespace {

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
  // x and y have no elements when M = 0 and may then be null
  if (w == nullptr || (M > 0 && (x == nullptr || y == nullptr))) return SP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return SP_ERR_MISALIGNED;
  if (M == 0) return SP_OK;
  GemmArgs g{x, w, y, in, in, out, M, out, in, false, false, false, status_word()};
  return launch_gemm(g, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

sp_status sp_linear_bwd(const void* dy, const void* x, const void* w, void* dx, void* dw, int M,
                        int in, int out, int accumulate_dw, void* stream) {
  const sp_status st = check_linear(M, in, out);
  if (st != SP_OK) return st;
  // dy and x have no elements when M = 0 and may then be null
  if (w == nullptr || (M > 0 && (dy == nullptr || x == nullptr)) ||
      (dx == nullptr && dw == nullptr))
    return SP_ERR_INVALID_ARG;
  if (accumulate_dw != 0 && accumulate_dw != 1) return SP_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(w) || (dx && !aligned16(dx)) ||
      (dw && !aligned16(dw)))
    return SP_ERR_MISALIGNED;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {
    // no rows: dx has no elements and dy^T . x is the zero matrix, so a dW that is not
    // accumulated into is cleared (one accumulated into keeps its value)
    if (dw != nullptr && accumulate_dw == 0 &&
        cudaMemsetAsync(dw, 0, static_cast<size_t>(out) * in * 2, s) != cudaSuccess)
      return SP_ERR_CUDA;
    return SP_OK;
  }
  uint32_t* status = status_word();
  // dx[M][in] = dy[M][out] . W[out][in]: k = out; W read with n = in contiguous
  if (dx != nullptr) {
    GemmArgs g{dy, w, dx, out, in, in, M, in, out, false, true, false, status};
    if (launch_gemm(g, s) != cudaSuccess) return SP_ERR_CUDA;
  }
  // dW[out][in] (+)= dy^T . x: k = the M rows; dy read with m = out contiguous, x with
  // n = in contiguous
  if (dw != nullptr) {
    GemmArgs g{dy, x, dw, out, in, in, out, in, M, true, true, accumulate_dw != 0, status};
    if (launch_gemm(g, s) != cudaSuccess) return SP_ERR_CUDA;
  }
  return SP_OK;
}

}  // extern "C"
