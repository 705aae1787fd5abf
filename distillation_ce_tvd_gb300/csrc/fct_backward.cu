// Backward kernels of the fused CE + TVD loss and of plain cross-entropy.
//
// Method: PR #1384 analysis, section "Backward Pass": with p = softmax(s),
// q = softmax(t) and sign_v = sign(p_v - q_v),
//   d ce / d s_v  = p_v - 1[v == target]
//   d tvd / d s_v = 0.5 * p_v * (sign_v - sigma)     (softmax Jacobian of 0.5*sign)
// and the kernel reloads both rows, recomputes p, q and the sign from the
// saved lse values, and writes
//   grad_v = grad_ce * p_v + grad_tvd * 0.5 * p_v * (sign_v - sigma) - grad_ce * 1[v == target],
// with zero rows for ignore_index and a zero subgradient at ties.
//
// GB300 mapping: a pure stream (2 reads + 1 write per element) cut into
// units of (row, 1024 vectors) (2048 for cross-entropy alone, which reads one
// tensor); a persistent grid of resident CTAs walks the units.  Per element the coefficient of p is c0 + h*sign with per-row
// c0 = grad_ce - h*sigma and h = grad_tvd/2, and sign from two compares that
// yield 0 at ties, so the inner loop is two ex2, two compares, one subtract
// and two FMAs/multiplies.  Each element is read and then written by the
// same thread, which makes grad_student == student (in place) safe.
#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

namespace {

constexpr int kThreads = 256;
// Vectors per thread per unit, all loaded before any is used: 4 per tensor for
// the fused loss (student + teacher), 12 for cross-entropy alone and when the
// signs come from the forward's sign words (the teacher is then read only
// for rows with a tie).  Measured at 8192 x 151936 bf16: 8 vectors gave
// 0.775 ms for ce_backward and 0.809 ms with sign words, 12 gave 0.755 and
// 0.775, 16 gave 0.759 and 0.847.
template <bool kTwo>
constexpr int kUnrollOf = kTwo ? 4 : 12;
template <bool kTwo>
constexpr int64_t kSegOf = int64_t(kThreads) * kUnrollOf<kTwo>;  // vectors per unit

// kSigns: the sign of p - q comes from the forward's sign words (a byte of
// bits per vector) for rows whose tie flag is clear; the coefficient of p is
// then fmaf(h, +-1, c0), the very values the sign expression gives, so the
// gradient is bit-identical.  Rows with a tie, and the ragged tail, recompute
// the sign from the teacher.
template <typename T, int VE, bool kTvd, bool kSigns = false>
__global__ void __launch_bounds__(kThreads) backward_kernel(BwdArgs a) {
  static_assert(!kSigns || (kTvd && VE > 1), "sign words cover the fused loss's vectors");
  constexpr int kUnroll = kUnrollOf<kTvd && !kSigns>;
  constexpr int64_t kSeg = kSegOf<kTvd && !kSigns>;
  const T* S = static_cast<const T*>(a.student);
  const T* Tt = static_cast<const T*>(a.teacher);
  T* G = static_cast<T*>(a.grad);
  const int64_t nvec = a.V / VE;
  const int64_t tail0 = nvec * VE;
  const int64_t nseg = nvec > 0 ? (nvec + kSeg - 1) / kSeg : 1;
  const int64_t units = a.BT * nseg;
  const uint64_t drop = policy_evict_first();

  for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int64_t row = unit / nseg;
    const int64_t seg = unit - row * nseg;
    const bool last_seg = (seg == nseg - 1);
    const int64_t v0 = seg * kSeg;
    const int64_t v1 = min(nvec, v0 + kSeg);
    const int64_t tg_full = a.target[row];
    const int64_t tg = tg_full - a.tg_base;  // in this row's columns (a vocabulary shard's)
    const T* srow = S + row * a.ld_s;
    const T* trow = kTvd ? Tt + row * a.ld_t : nullptr;
    T* grow = G + row * a.ld_g;

    const bool ignored = (tg_full == a.ignore_index);
    const int64_t v_all = a.V_full > 0 ? a.V_full : a.V;
    if (ignored || tg_full < 0 || tg_full >= v_all) {
      // Ignored rows get a zero gradient; out-of-range targets get NaN and
      // raise the status bit.  Neither reads the logits.
      const float fill = ignored ? 0.f : __uint_as_float(0x7fc00000u);
      if (!ignored && seg == 0 && threadIdx.x == 0 && a.dev_status)
        atomicOr(a.dev_status, FCT_DEV_TARGET_OUT_OF_RANGE);
      float f[VE];
#pragma unroll
      for (int j = 0; j < VE; ++j) f[j] = fill;
      for (int64_t i = v0 + threadIdx.x; i < v1; i += kThreads) store_vec<T, VE>(grow + i * VE, f, drop);
      if (last_seg && tail0 + threadIdx.x < a.V) Elem<T>::store1(grow + tail0 + threadIdx.x, fill);
      continue;
    }

    const float gce = a.grad_ce[row * a.grad_stride];
    const float ns2 = -(a.lse_s[row] * kLog2e);
    // coefficient of p: c = gce + h * (sign - sigma) = c0 + h * sign
    float nt2 = 0.f, h = 0.f, c0 = gce;
    if constexpr (kTvd) {
      h = 0.5f * a.grad_tvd[row * a.grad_stride];
      nt2 = -(a.lse_t[row] * kLog2e);
      c0 = gce - h * a.sigma[row];
    }

    auto grad_of = [&](const float (&xs)[VE], const float (&xt)[VE], int64_t base, float (&g)[VE]) {
#pragma unroll
      for (int j = 0; j < VE; ++j) {
        const float p = ex2(fmaf(xs[j], kLog2e, ns2));
        float c = gce;
        if constexpr (kTvd) c = fmaf(h, sgn_pq(p, ex2(fmaf(xt[j], kLog2e, nt2))), c0);
        g[j] = p * c;
      }
      const int64_t off = tg - base;
      if (static_cast<uint64_t>(off) < static_cast<uint64_t>(VE)) {
#pragma unroll
        for (int j = 0; j < VE; ++j)
          if (j == off) g[j] -= gce;
      }
    };

    int64_t i = v0 + threadIdx.x;
    bool from_bits = false;
    const uint8_t* brow = nullptr;
    if constexpr (kSigns) {
      brow = a.signs + row * a.ld_signs;
      from_bits = (*reinterpret_cast<const uint32_t*>(brow) == 0u);
    }
    if (kSigns && from_bits) {
      const float c_plus = fmaf(h, 1.f, c0), c_minus = fmaf(h, -1.f, c0);
      auto grad_bits = [&](const float (&xs)[VE], uint32_t bits, int64_t base, float (&g)[VE]) {
#pragma unroll
        for (int j = 0; j < VE; ++j) {
          const float p = ex2(fmaf(xs[j], kLog2e, ns2));
          g[j] = p * (((bits >> (VE - 1 - j)) & 1u) ? c_minus : c_plus);
        }
        const int64_t off = tg - base;
        if (static_cast<uint64_t>(off) < static_cast<uint64_t>(VE)) {
#pragma unroll
          for (int j = 0; j < VE; ++j)
            if (j == off) g[j] -= gce;
        }
      };
      const uint8_t* bits = brow + 4;
      if (i + (kUnroll - 1) * kThreads < v1) {
        uint4 rs[kUnroll];
        uint32_t sb[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
          rs[k] = load_raw<T, VE>(srow + (i + k * kThreads) * VE, drop);
          sb[k] = bits[i + k * kThreads];
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
          float xs[VE], g[VE];
          unpack_raw<T, VE>(rs[k], xs);
          grad_bits(xs, sb[k], (i + k * kThreads) * VE, g);
          store_vec<T, VE>(grow + (i + k * kThreads) * VE, g, drop);
        }
      } else {
        for (; i < v1; i += kThreads) {
          float xs[VE], g[VE];
          unpack_raw<T, VE>(load_raw<T, VE>(srow + i * VE, drop), xs);
          grad_bits(xs, bits[i], i * VE, g);
          store_vec<T, VE>(grow + i * VE, g, drop);
        }
      }
    } else if (!kSigns && i + (kUnroll - 1) * kThreads < v1) {  // full unit: all loads first
      // (with sign words only rows with a tie come here: the plain loop below
      // serves them and keeps the register count of the common case down)
      uint4 rs[kUnroll], rt[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        rs[k] = load_raw<T, VE>(srow + (i + k * kThreads) * VE, drop);
        if constexpr (kTvd) rt[k] = load_raw<T, VE>(trow + (i + k * kThreads) * VE, drop);
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        float xs[VE], xt[VE], g[VE];
        unpack_raw<T, VE>(rs[k], xs);
        if constexpr (kTvd) unpack_raw<T, VE>(rt[k], xt);
        grad_of(xs, xt, (i + k * kThreads) * VE, g);
        store_vec<T, VE>(grow + (i + k * kThreads) * VE, g, drop);
      }
    } else {
      for (; i < v1; i += kThreads) {
        float xs[VE], xt[VE], g[VE];
        unpack_raw<T, VE>(load_raw<T, VE>(srow + i * VE, drop), xs);
        if constexpr (kTvd) unpack_raw<T, VE>(load_raw<T, VE>(trow + i * VE, drop), xt);
        grad_of(xs, xt, i * VE, g);
        store_vec<T, VE>(grow + i * VE, g, drop);
      }
    }
    if (last_seg && tail0 + threadIdx.x < a.V) {
      const int64_t v = tail0 + threadIdx.x;
      float xs[1] = {Elem<T>::load1(srow + v)}, xt[1] = {0.f}, g[1];
      if constexpr (kTvd) xt[0] = Elem<T>::load1(trow + v);
      // one element: reuse the vector code with VE = 1 semantics
      const float p = ex2(fmaf(xs[0], kLog2e, ns2));
      float c = gce;
      if constexpr (kTvd) c = fmaf(h, sgn_pq(p, ex2(fmaf(xt[0], kLog2e, nt2))), c0);
      g[0] = p * c;
      if (v == tg) g[0] -= gce;
      Elem<T>::store1(grow + v, g[0]);
    }
  }
}

// Resident CTAs per SM of one backward configuration, queried once per device.
template <typename T, int VE, bool kTvd, bool kSigns>
int blocks_per_sm() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, backward_kernel<T, VE, kTvd, kSigns>,
                                                      kThreads, 0) != cudaSuccess) {
      cudaGetLastError();
      n = 1;
    }
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

template <typename T, int VE, bool kTvd, bool kSigns = false>
cudaError_t go(const BwdArgs& a, int sms, cudaStream_t st) {
  constexpr int64_t kSeg = kSegOf<kTvd && !kSigns>;
  const int64_t nvec = a.V / VE;
  const int64_t nseg = nvec > 0 ? (nvec + kSeg - 1) / kSeg : 1;
  const int64_t units = a.BT * nseg;
  int64_t grid = int64_t(sms) * blocks_per_sm<T, VE, kTvd, kSigns>();
  if (grid > units) grid = units;
  backward_kernel<T, VE, kTvd, kSigns><<<static_cast<unsigned>(grid), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdArgs& a, bool vec, int sms, cudaStream_t st) {
  const bool tvd = a.teacher != nullptr;
  if (a.signs) {  // sign words: vector path of the fused loss only
    if (!vec || !tvd) return cudaErrorInvalidValue;
    return a.dtype == FCT_BF16 ? go<bf16_t, 8, true, true>(a, sms, st)
                               : go<float, 4, true, true>(a, sms, st);
  }
  if (a.dtype == FCT_BF16) {
    if (tvd) return vec ? go<bf16_t, 8, true>(a, sms, st) : go<bf16_t, 1, true>(a, sms, st);
    return vec ? go<bf16_t, 8, false>(a, sms, st) : go<bf16_t, 1, false>(a, sms, st);
  }
  if (tvd) return vec ? go<float, 4, true>(a, sms, st) : go<float, 1, true>(a, sms, st);
  return vec ? go<float, 4, false>(a, sms, st) : go<float, 1, false>(a, sms, st);
}

}  // namespace fct
