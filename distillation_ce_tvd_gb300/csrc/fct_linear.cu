// Fused-linear CE + TVD, chunked over rows.
//
// The loss of the PR #1384 analysis takes logits; a model produces them as
// hidden states times an lm_head weight.  Materialising the (BT, V) logits
// of student and teacher costs 2*BT*V elements of memory and traffic.  Here
// the rows go through in blocks of R: per block, two plain GEMMs (cuBLAS,
// bf16 inputs, fp32 accumulate and output) write the block's student and
// teacher logits into the caller's workspace, the single-launch forward +
// backward kernel turns the student block into its gradient in place, a
// conversion kernel rounds that gradient to bf16, and two more GEMMs give the
// block's d loss / d hidden and accumulate d loss / d weight.  Only
// 2*R*V fp32 logits exist at a time.  The teacher is frozen (no gradients).
#include <cublas_v2.h>

#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

namespace {

constexpr int kConvThreads = 256;

// fp32 (rows, cols) with stride ld_src -> bf16 with stride ld_dst, rounded to
// nearest even.  8 elements per thread per iteration when both strides and
// bases allow 32/16-byte accesses (the workspace layout guarantees it).
__global__ void __launch_bounds__(kConvThreads) f32_to_bf16(const float* src, int64_t ld_src,
                                                            uint16_t* dst, int64_t ld_dst,
                                                            int64_t rows, int64_t cols) {
  const int64_t per_row = cols / 8;
  const int64_t total = rows * per_row;
  for (int64_t i = blockIdx.x * int64_t(kConvThreads) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kConvThreads) {
    const int64_t r = i / per_row, c = (i - r * per_row) * 8;
    const float4 a = *reinterpret_cast<const float4*>(src + r * ld_src + c);
    const float4 b = *reinterpret_cast<const float4*>(src + r * ld_src + c + 4);
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    *reinterpret_cast<uint4*>(dst + r * ld_dst + c) = o;
  }
  // ragged columns (cols % 8), one element per thread
  const int64_t tail = cols - per_row * 8;
  if (tail) {
    for (int64_t i = blockIdx.x * int64_t(kConvThreads) + threadIdx.x; i < rows * tail;
         i += int64_t(gridDim.x) * kConvThreads) {
      const int64_t r = i / tail, c = per_row * 8 + (i - r * tail);
      dst[r * ld_dst + c] = static_cast<uint16_t>(pack_bf16x2(src[r * ld_src + c], 0.f) & 0xffffu);
    }
  }
}

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

size_t linear_workspace_bytes(int64_t V, int64_t chunk_rows) {
  return size_t(2) * size_t(chunk_rows) * size_t(linear_logits_ld(V)) * sizeof(float);
}

cudaError_t launch_linear(const LinArgs& a, const FwdPlan& plan, int device, int sms,
                          cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_blas_mu);  // one cuBLAS handle per device, one caller at a time
  if (g_blas[device] == nullptr && cublasCreate(&g_blas[device]) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorInitializationError;
  cublasHandle_t h = g_blas[device];
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return cudaErrorInvalidValue;
  if (cublasSetMathMode(h, CUBLAS_DEFAULT_MATH) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorInvalidValue;

  const int64_t ldl = linear_logits_ld(a.V);  // fp32 logits rows: 32-byte multiple
  float* Ls = static_cast<float*>(a.workspace);
  float* Lt = Ls + a.chunk_rows * ldl;
  uint16_t* G = reinterpret_cast<uint16_t*>(Lt);  // bf16 gradient reuses the teacher block
  const int64_t ldg = ldl;
  const auto* Hs = static_cast<const uint16_t*>(a.h_s);
  const auto* Ht = static_cast<const uint16_t*>(a.h_t);

  for (int64_t r0 = 0; r0 < a.BT; r0 += a.chunk_rows) {
    const int64_t R = (a.BT - r0 < a.chunk_rows) ? a.BT - r0 : a.chunk_rows;
    // logits (row-major R x V) = H (R x D) * W^T, as column-major V x R
    if (gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, a.V, R, a.d_s, a.w_s, a.ld_ws, Hs + r0 * a.ld_hs,
             a.ld_hs, 0.f, Ls, CUDA_R_32F, ldl) != CUBLAS_STATUS_SUCCESS)
      return cudaErrorLaunchFailure;
    if (gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, a.V, R, a.d_t, a.w_t, a.ld_wt, Ht + r0 * a.ld_ht,
             a.ld_ht, 0.f, Lt, CUDA_R_32F, ldl) != CUBLAS_STATUS_SUCCESS)
      return cudaErrorLaunchFailure;
    // the loss on the block, its logit gradient written over Ls
    FwdArgs f{Ls, Lt, ldl, ldl, FCT_F32, a.target + r0, R, a.V, a.ignore_index,
              a.ce + r0, a.tvd + r0, a.lse_s + r0, a.lse_t + r0, a.sigma + r0, a.dev_status,
              Ls, ldl, a.grad_ce + (a.grad_stride ? r0 : 0),
              a.grad_tvd + (a.grad_stride ? r0 : 0), a.grad_stride, plan.keep_normal ? 1 : 0};
    cudaError_t e = launch_forward(f, plan, st);
    if (e != cudaSuccess) return e;
    if (a.grad_h_s == nullptr && a.grad_w_s == nullptr) continue;
    int64_t blocks = (R * (a.V / 8) + kConvThreads - 1) / kConvThreads;
    if (blocks > int64_t(sms) * 8) blocks = int64_t(sms) * 8;
    if (blocks < 1) blocks = 1;
    f32_to_bf16<<<static_cast<unsigned>(blocks), kConvThreads, 0, st>>>(Ls, ldl, G, ldg, R, a.V);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
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
