// Forward kernels of the fused CE + TVD loss and of plain cross-entropy.
//
// Method: PR #1384 analysis ("[Liger-Kernel] Liger-Kernel: Cross-Entropy와
// Total Variation Distance를 하나로 융합하여 성능을 극대화하다"), section
// "Forward Pass": step 1 streams each row once for the online max / sum-exp
// of student and teacher, step 2 streams it again for
// 0.5*sum|p - q| and sigma = sum p*sign(p - q), then five per-row stores.
//
// GB300 mapping
//   * A row is owned by a thread-block cluster of C CTAs (C in {1,2,4,8});
//     each CTA streams a contiguous 1/C of the row's 16-byte vectors.  The
//     CTAs exchange only scalar partials, through distributed shared memory.
//   * Step 1 reads the row from HBM with an L2 evict_last hint; step 2
//     re-reads the same bytes, which are still in L2 because the number of
//     rows in flight (clusters on the GPU) times the row size is kept well
//     under the L2 capacity by the choice of C.  HBM therefore sees each
//     logit about once, and no (BT, V) buffer is ever written.
//   * The grid is persistent: one cluster per slot the GPU can hold, looping
//     over rows, so the launch is sized by the SM count, not by BT.
//   * Student and teacher go through the very same code, so a row whose
//     teacher equals its student bit for bit gets p == q everywhere and
//     tvd = sigma = 0 exactly.
#include <cooperative_groups.h>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace cg = cooperative_groups;

namespace fct {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;  // 16-byte loads in flight per thread and row

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Block-wide merge of two Lse2 states.  Every warp folds the per-warp
// partials in the same order, so every thread ends with identical values.
// `buf` must not be rewritten before the next __syncthreads of the caller.
__device__ __forceinline__ void block_merge2(Lse2& a, Lse2& b, float4* buf) {
  a = warp_merge(a);
  b = warp_merge(b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_float4(a.m2, a.s, b.m2, b.s);
  __syncthreads();
  float4 w = (lane < kWarps) ? buf[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  a = warp_merge(Lse2{w.x, w.y});
  b = warp_merge(Lse2{w.z, w.w});
}

__device__ __forceinline__ void block_sum2(float& x, float& y, float2* buf) {
  x = warp_sum(x);
  y = warp_sum(y);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_float2(x, y);
  __syncthreads();
  float2 w = (lane < kWarps) ? buf[lane] : make_float2(0.f, 0.f);
  x = warp_sum(w.x);
  y = warp_sum(w.y);
}

// Step-1 streaming over vectors [vb, ve) of one row (and of the teacher row
// when kTvd): thread i takes vectors vb+i, vb+i+kThreads, ...
template <typename T, int VE, bool kTvd>
__device__ __forceinline__ void lse_pass(const T* s, const T* t, int64_t vb, int64_t ve,
                                         uint64_t pol, Lse2& a, Lse2& b) {
  int64_t i = vb + threadIdx.x;
  for (; i + (kUnroll - 1) * kThreads < ve; i += kUnroll * kThreads) {
    uint4 rs[kUnroll], rt[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      rs[k] = load_raw<T, VE>(s + (i + k * kThreads) * VE, pol);
      if constexpr (kTvd) rt[k] = load_raw<T, VE>(t + (i + k * kThreads) * VE, pol);
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      float x[VE];
      unpack_raw<T, VE>(rs[k], x);
      lse2_update(a, x);
      if constexpr (kTvd) {
        unpack_raw<T, VE>(rt[k], x);
        lse2_update(b, x);
      }
    }
  }
  for (; i < ve; i += kThreads) {
    float x[VE];
    unpack_raw<T, VE>(load_raw<T, VE>(s + i * VE, pol), x);
    lse2_update(a, x);
    if constexpr (kTvd) {
      unpack_raw<T, VE>(load_raw<T, VE>(t + i * VE, pol), x);
      lse2_update(b, x);
    }
  }
}

// p and q of one element pair folded into (sum |p - q|, sum p*sign(p - q)).
__device__ __forceinline__ void tvd_accum(float xs, float xt, float ns2, float nt2,
                                          float& abs_sum, float& sig) {
  const float p = ex2(fmaf(xs, kLog2e, ns2));
  const float q = ex2(fmaf(xt, kLog2e, nt2));
  const float d = p - q;
  abs_sum += fabsf(d);
  sig += (d > 0.f) ? p : ((d < 0.f) ? -p : 0.f);
}

template <typename T, int VE>
__device__ __forceinline__ void tvd_pass(const T* s, const T* t, int64_t vb, int64_t ve,
                                         uint64_t pol, float ns2, float nt2,
                                         float& abs_sum, float& sig) {
  int64_t i = vb + threadIdx.x;
  for (; i + (kUnroll - 1) * kThreads < ve; i += kUnroll * kThreads) {
    uint4 rs[kUnroll], rt[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      rs[k] = load_raw<T, VE>(s + (i + k * kThreads) * VE, pol);
      rt[k] = load_raw<T, VE>(t + (i + k * kThreads) * VE, pol);
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      float xs[VE], xt[VE];
      unpack_raw<T, VE>(rs[k], xs);
      unpack_raw<T, VE>(rt[k], xt);
      float a = 0.f, g = 0.f;
#pragma unroll
      for (int j = 0; j < VE; ++j) tvd_accum(xs[j], xt[j], ns2, nt2, a, g);
      abs_sum += a;
      sig += g;
    }
  }
  for (; i < ve; i += kThreads) {
    float xs[VE], xt[VE];
    unpack_raw<T, VE>(load_raw<T, VE>(s + i * VE, pol), xs);
    unpack_raw<T, VE>(load_raw<T, VE>(t + i * VE, pol), xt);
    float a = 0.f, g = 0.f;
#pragma unroll
    for (int j = 0; j < VE; ++j) tvd_accum(xs[j], xt[j], ns2, nt2, a, g);
    abs_sum += a;
    sig += g;
  }
}

// One row per cluster of C CTAs; kTvd = false is the plain cross-entropy
// forward (student only, ce and lse outputs).
template <typename T, int VE, int C, bool kTvd>
__global__ void __launch_bounds__(kThreads, 1) forward_kernel(FwdArgs p) {
  __shared__ float4 red_lse[kWarps];
  __shared__ float2 red_sum[kWarps];
  __shared__ float4 part_lse;  // this CTA's step-1 partial, read by its peers
  __shared__ float2 part_sum;  // this CTA's step-2 partial, read by rank 0

  const T* __restrict__ S = static_cast<const T*>(p.student);
  const T* __restrict__ Tt = static_cast<const T*>(p.teacher);
  const int rank = (C > 1) ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
  const int64_t cluster_id = blockIdx.x / C;
  const int64_t n_clusters = gridDim.x / C;

  const int64_t nvec = p.V / VE;
  const int64_t tail0 = nvec * VE;
  const int64_t per = (nvec + C - 1) / C;
  const int64_t vb = min(nvec, rank * per);
  const int64_t ve = min(nvec, vb + per);
  const bool owns_tail = (rank == C - 1);

  const uint64_t keep = policy_evict_last();
  const uint64_t drop = policy_evict_first();

  for (int64_t row = cluster_id; row < p.BT; row += n_clusters) {
    const int64_t tg = p.target[row];
    if (tg == p.ignore_index) {
      if (rank == 0 && threadIdx.x == 0) {
        p.ce[row] = 0.f;
        p.lse_s[row] = 0.f;
        if constexpr (kTvd) {
          p.tvd[row] = 0.f;
          p.lse_t[row] = 0.f;
          p.sigma[row] = 0.f;
        }
      }
      continue;  // uniform over the whole cluster: no barrier is skipped unevenly
    }
    const T* srow = S + row * p.ld_s;
    const T* trow = kTvd ? Tt + row * p.ld_t : nullptr;

    // ---- step 1: log-sum-exp of both rows
    Lse2 a = lse2_empty(), b = lse2_empty();
    lse_pass<T, VE, kTvd>(srow, trow, vb, ve, kTvd ? keep : drop, a, b);
    if (owns_tail && tail0 + threadIdx.x < p.V) {
      float xs[1] = {Elem<T>::load1(srow + tail0 + threadIdx.x)};
      lse2_update(a, xs);
      if constexpr (kTvd) {
        float xt[1] = {Elem<T>::load1(trow + tail0 + threadIdx.x)};
        lse2_update(b, xt);
      }
    }
    block_merge2(a, b, red_lse);
    if constexpr (C > 1) {
      if (threadIdx.x == 0) part_lse = make_float4(a.m2, a.s, b.m2, b.s);
      cluster_sync_all();
      cg::cluster_group cl = cg::this_cluster();
      a = lse2_empty();
      b = lse2_empty();
#pragma unroll
      for (int r = 0; r < C; ++r) {  // same order in every CTA: identical results
        const float4 w = *cl.map_shared_rank(&part_lse, r);
        a = lse2_merge(a, Lse2{w.x, w.y});
        b = lse2_merge(b, Lse2{w.z, w.w});
      }
    }
    const float lse_s = lse2_finish(a);

    if constexpr (!kTvd) {
      if (rank == 0 && threadIdx.x == 0) {
        p.lse_s[row] = lse_s;
        if (tg < 0 || tg >= p.V) {
          p.ce[row] = __uint_as_float(0x7fc00000u);
          if (p.dev_status) atomicOr(p.dev_status, FCT_DEV_TARGET_OUT_OF_RANGE);
        } else {
          p.ce[row] = lse_s - Elem<T>::load1(srow + tg);
        }
      }
      // Peers may still read part_lse and warps may still read red_lse.
      if constexpr (C > 1) {
        cluster_sync_all();
      } else {
        __syncthreads();
      }
    } else {
      const float lse_t = lse2_finish(b);
      // The backward recomputes p and q from the stored lse values with this
      // same expression, so both passes see bit-identical p and q.
      const float ns2 = -(lse_s * kLog2e);
      const float nt2 = -(lse_t * kLog2e);

      // ---- step 2: sum |p - q| and sigma
      float abs_sum = 0.f, sig = 0.f;
      tvd_pass<T, VE>(srow, trow, vb, ve, drop, ns2, nt2, abs_sum, sig);
      if (owns_tail && tail0 + threadIdx.x < p.V) {
        tvd_accum(Elem<T>::load1(srow + tail0 + threadIdx.x),
                  Elem<T>::load1(trow + tail0 + threadIdx.x), ns2, nt2, abs_sum, sig);
      }
      block_sum2(abs_sum, sig, red_sum);
      if constexpr (C > 1) {
        if (threadIdx.x == 0) part_sum = make_float2(abs_sum, sig);
        cluster_sync_all();
        if (rank == 0 && threadIdx.x == 0) {
          cg::cluster_group cl = cg::this_cluster();
          abs_sum = 0.f;
          sig = 0.f;
#pragma unroll
          for (int r = 0; r < C; ++r) {
            const float2 w = *cl.map_shared_rank(&part_sum, r);
            abs_sum += w.x;
            sig += w.y;
          }
        }
      }
      if (rank == 0 && threadIdx.x == 0) {
        p.tvd[row] = 0.5f * abs_sum;
        p.lse_s[row] = lse_s;
        p.lse_t[row] = lse_t;
        p.sigma[row] = sig;
        if (tg < 0 || tg >= p.V) {
          p.ce[row] = __uint_as_float(0x7fc00000u);
          if (p.dev_status) atomicOr(p.dev_status, FCT_DEV_TARGET_OUT_OF_RANGE);
        } else {
          p.ce[row] = lse_s - Elem<T>::load1(srow + tg);
        }
      }
    }
  }
  // No CTA may leave while a peer can still read its shared memory.
  if constexpr (C > 1) cluster_sync_all();
}

template <typename T, int VE, int C, bool kTvd>
cudaError_t launch(const FwdArgs& a, int n_clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_clusters * C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, forward_kernel<T, VE, C, kTvd>, a);
}

template <typename T, int VE, int C, bool kTvd>
int max_clusters() {
  static int cached = [] {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * 64);
    cfg.blockDim = dim3(kThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, forward_kernel<T, VE, C, kTvd>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    return n;
  }();
  return cached;
}

template <typename T, int VE, bool kTvd>
cudaError_t dispatch_c(const FwdArgs& a, int C, int n_slots, cudaStream_t st) {
  auto go = [&](auto cc) -> cudaError_t {
    constexpr int CC = decltype(cc)::value;
    int n = max_clusters<T, VE, CC, kTvd>();
    if (n <= 0) n = 1;
    if (n_slots > 0 && n > n_slots) n = n_slots;
    if (n > a.BT) n = static_cast<int>(a.BT);
    return launch<T, VE, CC, kTvd>(a, n, st);
  };
  switch (C) {
    case 1: return go(std::integral_constant<int, 1>{});
    case 2: return go(std::integral_constant<int, 2>{});
    case 4: return go(std::integral_constant<int, 4>{});
    default: return go(std::integral_constant<int, 8>{});
  }
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, const FwdPlan& plan, cudaStream_t st) {
  if (a.dtype == FCT_BF16) {
    if (a.tvd) {
      return plan.vec ? dispatch_c<bf16_t, 8, true>(a, plan.cluster, plan.slots, st)
                      : dispatch_c<bf16_t, 1, true>(a, plan.cluster, plan.slots, st);
    }
    return plan.vec ? dispatch_c<bf16_t, 8, false>(a, plan.cluster, plan.slots, st)
                    : dispatch_c<bf16_t, 1, false>(a, plan.cluster, plan.slots, st);
  }
  if (a.tvd) {
    return plan.vec ? dispatch_c<float, 4, true>(a, plan.cluster, plan.slots, st)
                    : dispatch_c<float, 1, true>(a, plan.cluster, plan.slots, st);
  }
  return plan.vec ? dispatch_c<float, 4, false>(a, plan.cluster, plan.slots, st)
                  : dispatch_c<float, 1, false>(a, plan.cluster, plan.slots, st);
}

}  // namespace fct
