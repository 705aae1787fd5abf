// Vocabulary-parallel CE + TVD: the loss when each device holds a column
// range (shard) of the student and teacher logits.
//
// Method: PR #1384 analysis, "Forward Pass" and "Backward Pass".  A row's
// log-sum-exp, its TVD and sigma are sums over the vocabulary, so they split
// into per-shard partial sums that merge exactly (up to rounding order):
//   pass 1, per shard k: lse_k of the student and of the teacher over the
//           shard's columns, and the student logit at the target when the
//           shard holds it;
//   merge:  lse = log sum_k exp(lse_k) for each tensor, ce = lse_s - s[target];
//   pass 2, per shard: sum p*sign(p - q) and sum q*sign(p - q) over the shard,
//           p and q from the merged lse values (the sign of p - q needs both);
//   merge:  sigma = sum_k sigma_k, sum |p - q| = sum_k (sigma_k - tau_k);
//   pass 3, per shard: the backward kernel on the shard's columns with the
//           merged lse and sigma (launch_backward with a shard offset).
// Between the passes the partials (3 and 2 floats per row and shard) are
// exchanged by the caller (an all-gather across the devices that hold the
// shards); the merges take the shards in shard order, so every device gets
// bit-identical merged values.  Distributing a model's vocabulary this way is
// this library's addition; the per-element arithmetic is that of the fused
// kernels (base 2, ex2, the same tie rule).
//
// GB300 mapping: passes 1 and 2 are one CTA of 256 threads per row
// (persistent over rows, as many CTAs as are resident at once), 16-byte
// vector loads (4 in flight per thread per tensor) when the shard's columns
// start on 16 bytes, plain element loads otherwise, fp32 accumulation,
// warp-shuffle and shared-memory reductions.  The merges are one thread per
// row.
#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

namespace {

constexpr int kVpThreads = 256;
constexpr int kVpUnroll = 4;

// Block-wide merge of two Lse2 states (same fold order in every thread).
__device__ __forceinline__ void vp_block_merge2(Lse2& a, Lse2& b, float4* buf) {
  constexpr int kWarps = kVpThreads / 32;
  a = warp_merge(a);
  b = warp_merge(b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_float4(a.m2, a.s, b.m2, b.s);
  __syncthreads();
  const float4 w = (lane < kWarps) ? buf[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  a = warp_merge(Lse2{w.x, w.y});
  b = warp_merge(Lse2{w.z, w.w});
  __syncthreads();  // buf is reused by the next row
}

__device__ __forceinline__ void vp_block_sum2(float& x, float& y, float2* buf) {
  constexpr int kWarps = kVpThreads / 32;
  x = warp_sum(x);
  y = warp_sum(y);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_float2(x, y);
  __syncthreads();
  const float2 w = (lane < kWarps) ? buf[lane] : make_float2(0.f, 0.f);
  x = warp_sum(w.x);
  y = warp_sum(w.y);
  __syncthreads();
}

// Pass 1: per row, the shard's lse of student and teacher and the student
// logit at the target (0 when the target is not in this shard).
template <typename T, int VE>
__global__ void __launch_bounds__(kVpThreads) vp_lse_kernel(VpArgs a) {
  __shared__ float4 buf[kVpThreads / 32];
  // the element loop takes every column on the scalar path (VE == 1), the
  // ragged tail after the last full vector otherwise
  const int64_t nvec = a.V / VE, tail0 = (VE > 1) ? nvec * VE : 0;
  const uint64_t pol = policy_evict_first();
  for (int64_t row = blockIdx.x; row < a.BT; row += gridDim.x) {
    const int64_t tg = a.target[row];
    float* out = a.part + row * 3;
    if (tg == a.ignore_index) {
      if (threadIdx.x == 0) out[0] = out[1] = out[2] = 0.f;
      continue;
    }
    const T* srow = static_cast<const T*>(a.student) + row * a.ld_s;
    const T* trow = static_cast<const T*>(a.teacher) + row * a.ld_t;
    Lse2 fs = lse2_empty(), ft = lse2_empty();
    if constexpr (VE > 1) {
      Lse2x xs2 = lse2x_empty(), xt2 = lse2x_empty();
      int64_t v = threadIdx.x;
      for (; v + (kVpUnroll - 1) * kVpThreads < nvec; v += kVpUnroll * kVpThreads) {
        uint4 rs[kVpUnroll], rt[kVpUnroll];
#pragma unroll
        for (int k = 0; k < kVpUnroll; ++k) {
          rs[k] = load_raw<T, VE>(srow + (v + k * kVpThreads) * VE, pol);
          rt[k] = load_raw<T, VE>(trow + (v + k * kVpThreads) * VE, pol);
        }
#pragma unroll
        for (int k = 0; k < kVpUnroll; ++k) {
          float xs[VE], xt[VE];
          unpack_raw<T, VE>(rs[k], xs);
          unpack_raw<T, VE>(rt[k], xt);
          lse2x_update(xs2, xs);
          lse2x_update(xt2, xt);
        }
      }
      for (; v < nvec; v += kVpThreads) {
        float xs[VE], xt[VE];
        unpack_raw<T, VE>(load_raw<T, VE>(srow + v * VE, pol), xs);
        unpack_raw<T, VE>(load_raw<T, VE>(trow + v * VE, pol), xt);
        lse2x_update(xs2, xs);
        lse2x_update(xt2, xt);
      }
      fs = lse2x_fold(xs2);
      ft = lse2x_fold(xt2);
    }
    for (int64_t v = tail0 + threadIdx.x; v < a.V; v += kVpThreads) {
      float xs[1] = {Elem<T>::load1(srow + v)}, xt[1] = {Elem<T>::load1(trow + v)};
      lse2_update(fs, xs);
      lse2_update(ft, xt);
    }
    vp_block_merge2(fs, ft, buf);
    if (threadIdx.x == 0) {
      const int64_t rel = tg - a.v_begin;
      out[0] = lse2_finish(fs);
      out[1] = lse2_finish(ft);
      out[2] = (rel >= 0 && rel < a.V) ? Elem<T>::load1(srow + rel) : 0.f;
    }
  }
}

// Pass 2: per row, the shard's sum of p*sign(p - q) and of q*sign(p - q),
// with p and q from the merged lse values.
template <typename T, int VE>
__global__ void __launch_bounds__(kVpThreads) vp_tvd_kernel(VpArgs a) {
  __shared__ float2 buf[kVpThreads / 32];
  // the element loop takes every column on the scalar path (VE == 1), the
  // ragged tail after the last full vector otherwise
  const int64_t nvec = a.V / VE, tail0 = (VE > 1) ? nvec * VE : 0;
  const uint64_t pol = policy_evict_first();
  for (int64_t row = blockIdx.x; row < a.BT; row += gridDim.x) {
    float* out = a.part + row * 2;
    if (a.target[row] == a.ignore_index) {
      if (threadIdx.x == 0) out[0] = out[1] = 0.f;
      continue;
    }
    const T* srow = static_cast<const T*>(a.student) + row * a.ld_s;
    const T* trow = static_cast<const T*>(a.teacher) + row * a.ld_t;
    const float ns2 = -(a.lse_s[row] * kLog2e), nt2 = -(a.lse_t[row] * kLog2e);
    float sig = 0.f, tau = 0.f;
    auto one = [&](float xs, float xt) {
      const float p = ex2(fmaf(xs, kLog2e, ns2));
      const float q = ex2(fmaf(xt, kLog2e, nt2));
      const float sg = sgn_pq(p, q);
      sig = fmaf(p, sg, sig);
      tau = fmaf(q, sg, tau);
    };
    if constexpr (VE > 1) {
      int64_t v = threadIdx.x;
      for (; v + (kVpUnroll - 1) * kVpThreads < nvec; v += kVpUnroll * kVpThreads) {
        uint4 rs[kVpUnroll], rt[kVpUnroll];
#pragma unroll
        for (int k = 0; k < kVpUnroll; ++k) {
          rs[k] = load_raw<T, VE>(srow + (v + k * kVpThreads) * VE, pol);
          rt[k] = load_raw<T, VE>(trow + (v + k * kVpThreads) * VE, pol);
        }
#pragma unroll
        for (int k = 0; k < kVpUnroll; ++k) {
          float xs[VE], xt[VE];
          unpack_raw<T, VE>(rs[k], xs);
          unpack_raw<T, VE>(rt[k], xt);
#pragma unroll
          for (int j = 0; j < VE; ++j) one(xs[j], xt[j]);
        }
      }
      for (; v < nvec; v += kVpThreads) {
        float xs[VE], xt[VE];
        unpack_raw<T, VE>(load_raw<T, VE>(srow + v * VE, pol), xs);
        unpack_raw<T, VE>(load_raw<T, VE>(trow + v * VE, pol), xt);
#pragma unroll
        for (int j = 0; j < VE; ++j) one(xs[j], xt[j]);
      }
    }
    for (int64_t v = tail0 + threadIdx.x; v < a.V; v += kVpThreads)
      one(Elem<T>::load1(srow + v), Elem<T>::load1(trow + v));
    vp_block_sum2(sig, tau, buf);
    if (threadIdx.x == 0) {
      out[0] = sig;
      out[1] = tau;
    }
  }
}

// Merge of pass 1: per row, the shards' lse values (base-2 states with sum 1
// at their own maximum, folded in shard order), ce, zeros for ignored rows,
// NaN ce and the status bit for a target outside the vocabulary.
__global__ void vp_merge_lse_kernel(VpMergeArgs a) {
  for (int64_t row = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; row < a.BT;
       row += int64_t(gridDim.x) * blockDim.x) {
    const int64_t tg = a.target[row];
    if (tg == a.ignore_index) {
      a.ce[row] = a.lse_s[row] = a.lse_t[row] = 0.f;
      continue;
    }
    Lse2 s = lse2_empty(), t = lse2_empty();
    float s_tg = 0.f;
    for (int64_t k = 0; k < a.n_shards; ++k) {
      const float* part = a.parts + (k * a.BT + row) * 3;
      s = lse2_merge(s, Lse2{part[0] * kLog2e, 1.f});
      t = lse2_merge(t, Lse2{part[1] * kLog2e, 1.f});
      s_tg += part[2];  // one shard holds the target, the others add 0
    }
    const float lse_s = lse2_finish(s);
    a.lse_s[row] = lse_s;
    a.lse_t[row] = lse2_finish(t);
    if (tg < 0 || tg >= a.V) {
      a.ce[row] = __uint_as_float(0x7fc00000u);
      if (a.dev_status) atomicOr(a.dev_status, FCT_DEV_TARGET_OUT_OF_RANGE);
    } else {
      a.ce[row] = lse_s - s_tg;
    }
  }
}

// Merge of pass 2: sigma = sum_k sigma_k, tvd = 0.5 * sum_k (sigma_k - tau_k).
__global__ void vp_merge_tvd_kernel(VpMergeArgs a) {
  for (int64_t row = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; row < a.BT;
       row += int64_t(gridDim.x) * blockDim.x) {
    if (a.target[row] == a.ignore_index) {
      a.tvd[row] = a.sigma[row] = 0.f;
      continue;
    }
    float sig = 0.f, abs_sum = 0.f;
    for (int64_t k = 0; k < a.n_shards; ++k) {
      const float* part = a.parts + (k * a.BT + row) * 2;
      sig += part[0];
      abs_sum += part[0] - part[1];
    }
    a.sigma[row] = sig;
    a.tvd[row] = 0.5f * abs_sum;
  }
}

// Resident CTAs per SM of a pass kernel on the current device (its register
// count sets it), queried once per device.  The persistent grid is exactly
// that many CTAs per SM: with more, the CTAs beyond the resident ones start
// only as others finish and run their rows at the end at low occupancy
// (bf16 passes: 48 registers, 5 resident CTAs; the 2-shard step at 8192 x
// 151936 bf16 took 2.925 ms with a grid of 8 CTAs per SM and 2.710 ms with
// the resident count, 4096 x 256000 fp32 4.375 and 4.263 ms).
template <typename K>
int resident_per_sm(K kernel) {
  static std::mutex mu;
  static int value[64];
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kVpThreads, 0) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      n = 1;
    }
    value[dev] = n;
    done[dev] = true;
  }
  return value[dev];
}

template <typename K>
void launch_pass(K kernel, const VpArgs& a, int sms, cudaStream_t st) {
  int64_t g = int64_t(sms) * resident_per_sm(kernel);
  if (g > a.BT) g = a.BT;
  kernel<<<static_cast<unsigned>(g), kVpThreads, 0, st>>>(a);
}

}  // namespace

cudaError_t launch_vp_pass(const VpArgs& a, bool vec, bool tvd_pass, int sms, cudaStream_t st) {
  if (a.BT == 0) return cudaSuccess;
  if (a.dtype == FCT_BF16) {
    if (tvd_pass) {
      vec ? launch_pass(vp_tvd_kernel<bf16_t, 8>, a, sms, st)
          : launch_pass(vp_tvd_kernel<bf16_t, 1>, a, sms, st);
    } else {
      vec ? launch_pass(vp_lse_kernel<bf16_t, 8>, a, sms, st)
          : launch_pass(vp_lse_kernel<bf16_t, 1>, a, sms, st);
    }
  } else {
    if (tvd_pass) {
      vec ? launch_pass(vp_tvd_kernel<float, 4>, a, sms, st)
          : launch_pass(vp_tvd_kernel<float, 1>, a, sms, st);
    } else {
      vec ? launch_pass(vp_lse_kernel<float, 4>, a, sms, st)
          : launch_pass(vp_lse_kernel<float, 1>, a, sms, st);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_vp_merge(const VpMergeArgs& a, bool tvd_merge, cudaStream_t st) {
  if (a.BT == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (a.BT + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (tvd_merge) {
    vp_merge_tvd_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(a);
  } else {
    vp_merge_lse_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace fct
