// Fused-linear CE + TVD, chunked over rows.
//
// The loss of the PR #1384 analysis takes logits; a model produces them as
// hidden states times an lm_head weight.  Materialising the (BT, V) logits
// of student and teacher costs 2*BT*V elements of memory and traffic.  Here
// the rows go through in blocks of R: per block, two plain GEMMs (cuBLAS,
// bf16 inputs, fp32 accumulate) write the block's student and teacher logits
// into the caller's workspace, the single-launch forward + backward kernel
// reads them and writes the block's logit gradient as bf16, and two more
// GEMMs give the block's d loss / d hidden and accumulate d loss / d weight.
// The logit blocks are fp32 (the GEMMs' own precision), or bf16 (rounded once
// by the GEMM, as a model's bf16 lm_head produces them), which halves their
// bytes and lets the gradient overwrite the student block in place.  Only the
// block's logits and gradient exist at a time.  The teacher is frozen (no
// gradients).
#include <cublas_v2.h>

#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

namespace {

std::mutex g_blas_mu;
cublasHandle_t g_blas[64] = {};

cublasStatus_t gemm(cublasHandle_t h, cublasOperation_t ta, cublasOperation_t tb, int64_t m,
                    int64_t n, int64_t k, const void* A, int64_t lda, const void* B, int64_t ldb,
                    float beta, void* C, cudaDataType ctype, int64_t ldc) {
  const float alpha = 1.f;
  return cublasGemmEx(h, ta, tb, static_cast<int>(m), static_cast<int>(n), static_cast<int>(k),
                      &alpha, A, CUDA_R_16BF, static_cast<int>(lda), B, CUDA_R_16BF,
                      static_cast<int>(ldb), &beta, C, ctype, static_cast<int>(ldc),
                      CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
}

}  // namespace

int64_t linear_logits_ld(int64_t V) { return (V + 7) / 8 * 8; }

size_t linear_workspace_bytes(int64_t V, int64_t chunk_rows, int logits_dtype) {
  // fp32: student and teacher logits, then the bf16 logit gradient;
  // bf16: student and teacher logits, the gradient written over the student's
  const size_t per_entry = logits_dtype == FCT_BF16 ? 2 * sizeof(uint16_t)
                                                    : 2 * sizeof(float) + sizeof(uint16_t);
  return size_t(chunk_rows) * size_t(linear_logits_ld(V)) * per_entry;
}

cudaError_t launch_linear(const LinArgs& a, const FwdPlan& plan, int device, int sms,
                          cudaStream_t st) {
  (void)sms;
  std::lock_guard<std::mutex> lk(g_blas_mu);  // one cuBLAS handle per device, one caller at a time
  if (g_blas[device] == nullptr && cublasCreate(&g_blas[device]) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorInitializationError;
  cublasHandle_t h = g_blas[device];
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return cudaErrorInvalidValue;
  if (cublasSetMathMode(h, CUBLAS_DEFAULT_MATH) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorInvalidValue;

  // logit rows padded to a multiple of 8 elements: 16-byte (bf16) or 32-byte
  // (fp32) row strides, so the loss kernel's vector path applies
  const int64_t ldl = linear_logits_ld(a.V);
  const bool bf16 = a.logits_dtype == FCT_BF16;
  const int64_t block_bytes = a.chunk_rows * ldl * (bf16 ? 2 : 4);
  char* Ls = static_cast<char*>(a.workspace);
  char* Lt = Ls + block_bytes;
  // the bf16 logit gradient: over the student block (same type, in place) or
  // after the two fp32 blocks
  void* G = bf16 ? static_cast<void*>(Ls) : static_cast<void*>(Lt + block_bytes);
  const int64_t ldg = ldl;
  const cudaDataType ltype = bf16 ? CUDA_R_16BF : CUDA_R_32F;
  const auto* Hs = static_cast<const uint16_t*>(a.h_s);
  const auto* Ht = static_cast<const uint16_t*>(a.h_t);

  for (int64_t r0 = 0; r0 < a.BT; r0 += a.chunk_rows) {
    const int64_t R = (a.BT - r0 < a.chunk_rows) ? a.BT - r0 : a.chunk_rows;
    // logits (row-major R x V) = H (R x D) * W^T, as column-major V x R
    if (gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, a.V, R, a.d_s, a.w_s, a.ld_ws, Hs + r0 * a.ld_hs,
             a.ld_hs, 0.f, Ls, ltype, ldl) != CUBLAS_STATUS_SUCCESS)
      return cudaErrorLaunchFailure;
    if (gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, a.V, R, a.d_t, a.w_t, a.ld_wt, Ht + r0 * a.ld_ht,
             a.ld_ht, 0.f, Lt, ltype, ldl) != CUBLAS_STATUS_SUCCESS)
      return cudaErrorLaunchFailure;
    // the loss on the block; its logit gradient, as bf16, into G
    FwdArgs f{Ls, Lt, ldl, ldl, bf16 ? FCT_BF16 : FCT_F32, a.target + r0, R, a.V, a.ignore_index,
              a.ce + r0, a.tvd + r0, a.lse_s + r0, a.lse_t + r0, a.sigma + r0, a.dev_status,
              G, ldg, a.grad_ce + (a.grad_stride ? r0 : 0),
              a.grad_tvd + (a.grad_stride ? r0 : 0), a.grad_stride, plan.keep_normal ? 1 : 0,
              /*grad_bf16=*/bf16 ? 0 : 1};
    cudaError_t e = launch_forward(f, plan, st);
    if (e != cudaSuccess) return e;
    if (a.grad_h_s == nullptr && a.grad_w_s == nullptr) continue;
    // d hidden (row-major R x D) = G (R x V) * W (V x D), as column-major D x R
    if (a.grad_h_s &&
        gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, a.d_s, R, a.V, a.w_s, a.ld_ws, G, ldg, 0.f,
             static_cast<uint16_t*>(a.grad_h_s) + r0 * a.ld_ghs, CUDA_R_16BF,
             a.ld_ghs) != CUBLAS_STATUS_SUCCESS)
      return cudaErrorLaunchFailure;
    // d weight (row-major V x D, fp32) += G^T (V x R) * H (R x D), as column-major D x V
    if (a.grad_w_s &&
        gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, a.d_s, a.V, R, Hs + r0 * a.ld_hs, a.ld_hs, G, ldg, 1.f,
             a.grad_w_s, CUDA_R_32F, a.ld_gws) != CUBLAS_STATUS_SUCCESS)
      return cudaErrorLaunchFailure;
  }
  return cudaGetLastError();
}

}  // namespace fct
