// Device helpers shared by the fused CE + TVD kernels (sm_103a).
//
// Everything works in base 2: a logit x enters the exponentials as
// x * log2(e), so every exponential is one ex2 (MUFU) after one FFMA.
#pragma once

#include <type_traits>

#include <cuda_runtime.h>
#include <stdint.h>

namespace fct {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- math

// 2^x on the special-function unit (flushes denormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Running (max, sum) state of a log-sum-exp in base 2:
//   m2 = max_v x_v*log2(e)  (rounded product),  s = sum_v 2^(x_v*log2(e) - m2).
// lse2 = m2 + log2(s), and the natural lse = lse2 * ln 2.
struct Lse2 {
  float m2;
  float s;
};

__device__ __forceinline__ Lse2 lse2_empty() { return Lse2{-INFINITY, 0.f}; }

// Merge of two partial states.  Commutative bit for bit (max and the sum of
// two products are), so butterfly reductions leave every lane identical.
__device__ __forceinline__ Lse2 lse2_merge(Lse2 a, Lse2 b) {
  const float m = fmaxf(a.m2, b.m2);
  const float sa = (a.m2 == -INFINITY) ? 0.f : a.s * ex2(a.m2 - m);
  const float sb = (b.m2 == -INFINITY) ? 0.f : b.s * ex2(b.m2 - m);
  return Lse2{m, sa + sb};
}

// Natural-log lse of a finished state.
__device__ __forceinline__ float lse2_finish(Lse2 a) {
  return (a.m2 + log2f(a.s)) * kLn2;
}

// Fold N values into a running state: rescale once per group if the group
// raises the maximum, then add the group's exponentials.
template <int N>
__device__ __forceinline__ void lse2_update(Lse2& st, const float (&x)[N]) {
  float vm = x[0];
#pragma unroll
  for (int j = 1; j < N; ++j) vm = fmaxf(vm, x[j]);
  const float m2n = vm * kLog2e;
  if (m2n > st.m2) {
    st.s *= ex2(st.m2 - m2n);
    st.m2 = m2n;
  }
  const float neg = -st.m2;
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) acc += ex2(fmaf(x[j], kLog2e, neg));
  st.s += acc;
}

// ---------------------------------------------------------------- step-2 sums

// sign(p - q) as a float: +1, -1, or 0 exactly when p == q (the zero
// subgradient at ties), from two compares that write 1.0f / 0.0f.
__device__ __forceinline__ float sgn_pq(float p, float q) {
  float gt, lt;
  asm("set.gt.f32.f32 %0, %1, %2;" : "=f"(gt) : "f"(p), "f"(q));
  asm("set.lt.f32.f32 %0, %1, %2;" : "=f"(lt) : "f"(p), "f"(q));
  return gt - lt;
}

// sign(p - q) of two (p, q) pairs on the FMA pipe instead of four compares
// on the ALU pipe (which step 2 is bound by): d = p - q rounded once, then
// 2 sat(d * 2^126 + 1/2) - 1.  That is exactly +1 or -1 for |d| >= 2^-127,
// i.e. for every nonzero difference except a subnormal one, and exactly 0
// at p == q (the zero subgradient at ties).  A nonzero subnormal difference
// gives a value strictly between -1 and 1; its bit pattern then fails the
// callers' tie test like a tie does, so sign bits are never taken from it.
__device__ __forceinline__ float sat_ramp(float d) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, 0f7E800000, 0f3F000000;" : "=f"(r) : "f"(d));
  return r;
}
__device__ __forceinline__ float2 sgn_pq2(float2 p, float2 q) {
  const float2 d = __ffma2_rn(q, make_float2(-1.f, -1.f), p);
  return __ffma2_rn(make_float2(sat_ramp(d.x), sat_ramp(d.y)), make_float2(2.f, 2.f),
                    make_float2(-1.f, -1.f));
}

// max(a, b, c) in one instruction (sm_100+).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int N>
__device__ __forceinline__ float vec_max(const float (&x)[N]) {
  if constexpr (N == 8) {
    return max3(max3(x[0], x[1], x[2]), max3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
  } else if constexpr (N == 4) {
    return max3(x[0], x[1], fmaxf(x[2], x[3]));
  } else {
    float m = x[0];
#pragma unroll
    for (int j = 1; j < N; ++j) m = fmaxf(m, x[j]);
    return m;
  }
}

// Running base-2 log-sum-exp state with two partial sums (two independent
// accumulation chains).
struct Lse2x {
  float m2;
  float2 s;
};

__device__ __forceinline__ Lse2x lse2x_empty() { return Lse2x{-INFINITY, make_float2(0.f, 0.f)}; }

__device__ __forceinline__ Lse2 lse2x_fold(Lse2x a) { return Lse2{a.m2, a.s.x + a.s.y}; }

// Fold N (even) values: one rescale if the group raises the maximum, then
// N FMAs for the exponents, N ex2 and N adds into two chains.
template <int N>
__device__ __forceinline__ void lse2x_update(Lse2x& st, const float (&x)[N]) {
  static_assert(N % 2 == 0, "pairs");
  const float m2n = vec_max(x) * kLog2e;
  if (m2n > st.m2) {
    const float sc = ex2(st.m2 - m2n);
    st.s.x *= sc;
    st.s.y *= sc;
    st.m2 = m2n;
  }
  const float nm = -st.m2;
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    st.s.x += ex2(fmaf(x[j], kLog2e, nm));
    st.s.y += ex2(fmaf(x[j + 1], kLog2e, nm));
  }
}

// ---------------------------------------------------------------- memory

// L2 eviction-priority policies for the cache_hint loads below.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte global load that skips L1 and tags the L2 line with `pol`.
__device__ __forceinline__ uint4 ld16(const void* ptr, uint64_t pol) {
  uint4 r;
  asm volatile(
      "ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(ptr), "l"(pol));
  return r;
}

// 16-byte global store that skips L1 and tags the L2 line with `pol`.
__device__ __forceinline__ void st16(void* ptr, uint4 v, uint64_t pol) {
  asm volatile(
      "st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
      :
      : "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
      : "memory");
}

// Asynchronous 16-byte global -> shared copy (per thread, no registers),
// tagged with an L2 eviction policy; completion is tracked per thread with
// commit/wait groups.
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;"
               :
               : "r"(smem_dst), "l"(src), "l"(pol)
               : "memory");
}
// Four 16-byte copies, shared dst + kBase + i*kDst <- global src + i*kSrc
// (i = 0..3), with the constant offsets folded into the instructions'
// addresses instead of computed into registers per copy.
template <int kBase, int kDst, int kSrc>
__device__ __forceinline__ void cp_async16x4(uint32_t smem_dst, const void* src, uint64_t pol) {
  asm volatile(
      "cp.async.cg.shared.global.L2::cache_hint [%0+%3], [%1], 16, %2;\n\t"
      "cp.async.cg.shared.global.L2::cache_hint [%0+%4], [%1+%5], 16, %2;\n\t"
      "cp.async.cg.shared.global.L2::cache_hint [%0+%6], [%1+%7], 16, %2;\n\t"
      "cp.async.cg.shared.global.L2::cache_hint [%0+%8], [%1+%9], 16, %2;"
      :
      : "r"(smem_dst), "l"(src), "l"(pol), "n"(kBase), "n"(kBase + kDst), "n"(kSrc),
        "n"(kBase + 2 * kDst), "n"(2 * kSrc), "n"(kBase + 3 * kDst), "n"(3 * kSrc)
      : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Element-type traits.  A "vector" is the 16 bytes one thread moves at once:
// 8 bf16 or 4 fp32 values.  The scalar path (VE == 1) serves rows whose
// pointers or strides are not 16-byte aligned.
struct bf16_t {
  uint16_t bits;
};

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float load1(const float* p) { return *p; }
  __device__ __forceinline__ static void unpack(uint4 w, float (&x)[4]) {
    x[0] = __uint_as_float(w.x);
    x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z);
    x[3] = __uint_as_float(w.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&x)[4]) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                      __float_as_uint(x[2]), __float_as_uint(x[3]));
  }
  __device__ __forceinline__ static void store1(float* p, float v) { *p = v; }
  static constexpr uint32_t kNanBits = 0x7fc00000u;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  // cvt.rn.bf16x2.f32 d, a, b puts a in the upper half and b in the lower.
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <>
struct Elem<bf16_t> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float load1(const bf16_t* p) {
    const unsigned short b = *reinterpret_cast<const unsigned short*>(p);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  __device__ __forceinline__ static void unpack(uint4 w, float (&x)[8]) {
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xffff0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xffff0000u);
    x[4] = __uint_as_float(w.z << 16);
    x[5] = __uint_as_float(w.z & 0xffff0000u);
    x[6] = __uint_as_float(w.w << 16);
    x[7] = __uint_as_float(w.w & 0xffff0000u);
  }
  __device__ __forceinline__ static uint4 pack(const float (&x)[8]) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                      pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
  }
  __device__ __forceinline__ static void store1(bf16_t* p, float v) {
    const uint32_t two = pack_bf16x2(v, 0.f);
    *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(two & 0xffffu);
  }
  static constexpr uint32_t kNanBits = 0x7fc0u;
};

// Load VE consecutive elements starting at element `p` as floats.
template <typename T, int VE>
__device__ __forceinline__ void load_vec(const T* p, uint64_t pol, float (&x)[VE]) {
  if constexpr (VE == 1) {
    x[0] = Elem<T>::load1(p);
  } else {
    static_assert(VE == Elem<T>::kVec, "a vector is 16 bytes");
    Elem<T>::unpack(ld16(p, pol), x);
  }
}

// Raw 16-byte (or one-element) load, unpacked later: keeps the registers of
// several loads in flight at 4 per vector instead of VE floats.
template <typename T, int VE>
__device__ __forceinline__ uint4 load_raw(const T* p, uint64_t pol) {
  if constexpr (VE == 1) {
    uint4 r;
    r.x = __float_as_uint(Elem<T>::load1(p));
    r.y = r.z = r.w = 0u;
    return r;
  } else {
    static_assert(VE == Elem<T>::kVec, "a vector is 16 bytes");
    return ld16(p, pol);
  }
}

template <typename T, int VE>
__device__ __forceinline__ void unpack_raw(uint4 r, float (&x)[VE]) {
  if constexpr (VE == 1) {
    x[0] = __uint_as_float(r.x);
  } else {
    Elem<T>::unpack(r, x);
  }
}

template <typename T, int VE>
__device__ __forceinline__ void store_vec(T* p, const float (&x)[VE], uint64_t pol) {
  if constexpr (VE == 1) {
    Elem<T>::store1(p, x[0]);
  } else {
    st16(p, Elem<T>::pack(x), pol);
  }
}

// A gradient vector of VE values in the gradient's element type TG, from a
// logits vector of type T: the same 16-byte store when TG == T, an 8-byte
// store of 4 bf16 values for fp32 logits with a bf16 gradient.
__device__ __forceinline__ void st8(void* ptr, uint32_t a, uint32_t b, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;"
               :
               : "l"(ptr), "r"(a), "r"(b), "l"(pol)
               : "memory");
}

template <typename T, typename TG, int VE>
__device__ __forceinline__ void store_grad(TG* p, const float (&x)[VE], uint64_t pol) {
  if constexpr (std::is_same<T, TG>::value || VE == 1) {
    store_vec<TG, VE>(p, x, pol);
  } else {
    static_assert(std::is_same<T, float>::value && std::is_same<TG, bf16_t>::value && VE == 4,
                  "a bf16 gradient of fp32 logits");
    st8(p, pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pol);
  }
}

// ---------------------------------------------------------------- warp

// Warp-wide merge of Lse2 states: the maximum first, then each lane's sum
// rescaled once to it, then a plain sum.  Every butterfly step combines the
// same two values in both lanes with a commutative operation (max, add), so
// all lanes end with identical results.
__device__ __forceinline__ Lse2 warp_merge(Lse2 a) {
  float m = a.m2;
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
  float s = (a.m2 == -INFINITY) ? 0.f : a.s * ex2(a.m2 - m);
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
  return Lse2{m, s};
}

__device__ __forceinline__ float warp_sum(float a) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) a += __shfl_xor_sync(0xffffffffu, a, m);
  return a;
}

// ---------------------------------------------------------------- mbarriers
//
// Every wait is bounded: after kWaitLimitCycles of SM clock (about 2 s) it
// gives up and sets the caller's abort flag, so a kernel whose producer stalls
// returns (with an error bit) instead of hanging.

constexpr long long kWaitLimitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Whether the phase of `bar` with parity `parity` has completed (may suspend
// the thread for a short hardware-defined time before answering no).
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for a phase.  Gives up after kWaitLimitCycles (setting *abort)
// or at once when *abort is already set and `heed_abort`.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort,
                                            bool heed_abort) {
  const long long t0 = clock64();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (heed_abort && *abort) return false;
    if (mbar_try(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) break;
  }
  *abort = 1;
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          bool heed_abort = true) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort, heed_abort);
}

}  // namespace fct
