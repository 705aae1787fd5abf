// Mean-over-tokens front end of the fused CE + TVD loss.
//
// The kernels of the PR #1384 analysis store per-row ce and tvd ("Forward
// Pass") and take per-row upstream gradients ("Backward Pass"); the
// reduction to one loss is left to the caller.  These two small kernels give
// the usual one: loss = (alpha * sum ce + beta * sum tvd) / n over the n rows
// whose target is not ignore_index, and its upstream gradients
// d loss / d ce_r = alpha / n, d loss / d tvd_r = beta / n (broadcast scalars,
// zero when n = 0).  Both run in one CTA with a fixed reduction order, so the
// results are deterministic; they read O(BT) bytes.
#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

namespace {

constexpr int kThreads = 1024;

// Sums (of doubles) over the block in a fixed order; every thread gets them.
__device__ __forceinline__ void block_sum3(double& a, double& b, double& c, double3* buf) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, m);
    b += __shfl_xor_sync(0xffffffffu, b, m);
    c += __shfl_xor_sync(0xffffffffu, c, m);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_double3(a, b, c);
  __syncthreads();
  double3 w = (lane < kThreads / 32) ? buf[lane] : make_double3(0.0, 0.0, 0.0);
  a = w.x;
  b = w.y;
  c = w.z;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, m);
    b += __shfl_xor_sync(0xffffffffu, b, m);
    c += __shfl_xor_sync(0xffffffffu, c, m);
  }
}

__global__ void __launch_bounds__(kThreads) mean_kernel(LossArgs p) {
  __shared__ double3 buf[kThreads / 32];
  double n = 0.0, sce = 0.0, stvd = 0.0;
  for (int64_t r = threadIdx.x; r < p.BT; r += kThreads) {
    if (p.target[r] != p.ignore_index) {
      n += 1.0;
      if (p.ce) sce += static_cast<double>(p.ce[r]);
      if (p.tvd) stvd += static_cast<double>(p.tvd[r]);
    }
  }
  block_sum3(n, sce, stvd, buf);
  if (threadIdx.x == 0) {
    const double inv = n > 0.0 ? 1.0 / n : 0.0;
    if (p.loss) p.loss[0] = static_cast<float>((p.alpha * sce + p.beta * stvd) * inv);
    if (p.grad_ce) p.grad_ce[0] = static_cast<float>(p.alpha * inv);
    if (p.grad_tvd) p.grad_tvd[0] = static_cast<float>(p.beta * inv);
    if (p.count) p.count[0] = static_cast<int64_t>(n);
  }
}

}  // namespace

cudaError_t launch_mean(const LossArgs& a, cudaStream_t st) {
  mean_kernel<<<1, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fct
