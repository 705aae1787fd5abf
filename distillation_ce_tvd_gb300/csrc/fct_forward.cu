// Forward kernels of the fused CE + TVD loss and of plain cross-entropy.
//
// Method: PR #1384 analysis ("[Liger-Kernel] Liger-Kernel: Cross-Entropy와
// Total Variation Distance를 하나로 융합하여 성능을 극대화하다"), section
// "Forward Pass": step 1 streams each row once for the online max / sum-exp
// of student and teacher, step 2 streams it again for
// 0.5*sum|p - q| and sigma = sum p*sign(p - q), then five per-row stores.
//
// GB300 mapping
//   * A row is owned by one CTA of 512 threads or, when the rows in flight
//     would not fit L2 that way, by a thread-block cluster of C CTAs
//     (C in {2,4,8}); each CTA streams a contiguous 1/C of the row's 16-byte
//     vectors.  The CTAs exchange only scalar partials, through distributed
//     shared memory.
//   * Step 1 reads the row from HBM with an L2 evict_last hint; step 2
//     re-reads the same bytes, which are still in L2 because the number of
//     rows in flight (clusters on the GPU) times the row size is kept under
//     the L2 capacity.  HBM therefore sees each logit about once, and no
//     (BT, V) buffer is ever written.
//   * Every thread streams its own vectors through a private ring in shared
//     memory (kStages steps of kPerStep 16-byte vectors per tensor), filled
//     by cp.async kStages - 1 steps ahead of the step being read.  The feed
//     runs on across the pass boundaries and into the next row, so loads
//     stay in flight while the CTA reduces; no thread ever reads another
//     thread's slot, so the ring needs no barrier.
//   * Step 1 takes exponents against a running reference maximum and redoes a
//     step against a raised maximum only when its sum reaches 2^64, so the
//     common step costs one FMA, one ex2 and one add per element.
//   * Step 2 accumulates sigma = sum p*sign(p - q) and tau = sum q*sign(p - q)
//     with sign from two compares (0 at ties: zero subgradient); then
//     sum|p - q| = sigma - tau.
//   * The grid is persistent: one cluster per row slot, looping over rows.
//     When every cluster has many rows, the clusters start in interleaved
//     groups spread over about half a row's time (a one-off wait on the SM
//     clock before the first loads), so that their HBM-bound first passes do
//     not all fall at the same moments.
//   * With the upstream gradients known before the launch, a third pass over
//     the still L2-resident student row writes the student gradient of the
//     "Backward Pass" in the same launch (the single-launch forward +
//     backward), so HBM sees 2 reads and 1 write per element instead of 4
//     reads and 1 write.  Step 2 leaves each element's sign bit in shared
//     memory, so step 3 reads only the student (p from the student logit, the
//     coefficient of p picked by the bit); a thread that met an exact tie
//     recomputes the sign from the teacher instead.
//   * The forward alone can also store those sign bits in global memory (one
//     byte per vector after a per-row tie flag), so that the backward reads
//     the student and the bits instead of the teacher.
//   * Student and teacher go through the very same code, so a row whose
//     teacher equals its student bit for bit gets p == q everywhere and
//     tvd = sigma = 0 exactly.
#include <cooperative_groups.h>

#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace cg = cooperative_groups;

namespace fct {

namespace {

constexpr int kMaxWarps = 32;

// Cluster barrier.  Every exchange here has one writer per CTA (thread 0
// stores the CTA's partials in its own shared memory before the barrier; the
// peers read them after it), so only that thread fences its writes to
// cluster scope and every thread arrives relaxed: a release arrive by all
// threads made each of them wait for its own outstanding loads (the ring's
// copies in flight), measured as membar stalls.  Reads of peers' partials
// are consumed before the thread's next arrive, so the next write cannot
// overtake them.
__device__ __forceinline__ void cluster_sync_all() {
  if (threadIdx.x == 0) asm volatile("fence.acq_rel.cluster;" ::: "memory");
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Barrier of the NT threads that take part in a row's reductions: the whole
// CTA, or (kNamed) the consumer warps of a kernel whose producer warp runs on
// its own, on named barrier 1.
template <int NT, bool kNamed>
__device__ __forceinline__ void rows_sync() {
  if constexpr (kNamed) {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  } else {
    __syncthreads();
  }
}

// Block-wide merge of two Lse2 states.  Every warp folds the per-warp
// partials in the same order, so every thread ends with identical values.
// `buf` must not be rewritten before the caller's next barrier.
template <int NT, bool kNamed = false>
__device__ __forceinline__ void block_merge2(Lse2& a, Lse2& b, float4* buf) {
  constexpr int kWarps = NT / 32;
  a = warp_merge(a);
  b = warp_merge(b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_float4(a.m2, a.s, b.m2, b.s);
  rows_sync<NT, kNamed>();
  float4 w = (lane < kWarps) ? buf[lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
  a = warp_merge(Lse2{w.x, w.y});
  b = warp_merge(Lse2{w.z, w.w});
}

template <int NT, bool kNamed = false>
__device__ __forceinline__ void block_sum2(float& x, float& y, float2* buf) {
  constexpr int kWarps = NT / 32;
  x = warp_sum(x);
  y = warp_sum(y);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) buf[warp] = make_float2(x, y);
  rows_sync<NT, kNamed>();
  float2 w = (lane < kWarps) ? buf[lane] : make_float2(0.f, 0.f);
  x = warp_sum(w.x);
  y = warp_sum(w.y);
}

// The C CTAs of a cluster fold their step-1 partials in rank order.
template <int C>
__device__ __forceinline__ void cluster_merge2(Lse2& a, Lse2& b, float4* part) {
  if constexpr (C > 1) {
    if (threadIdx.x == 0) *part = make_float4(a.m2, a.s, b.m2, b.s);
    cluster_sync_all();
    cg::cluster_group cl = cg::this_cluster();
    a = lse2_empty();
    b = lse2_empty();
#pragma unroll
    for (int r = 0; r < C; ++r) {
      const float4 w = *cl.map_shared_rank(part, r);
      a = lse2_merge(a, Lse2{w.x, w.y});
      b = lse2_merge(b, Lse2{w.z, w.w});
    }
  }
}

// Rank 0 (thread 0) folds the step-2 partials of the C CTAs in rank order.
template <int C>
__device__ __forceinline__ void cluster_sum2(float& x, float& y, float2* part, int rank) {
  if constexpr (C > 1) {
    if (threadIdx.x == 0) *part = make_float2(x, y);
    cluster_sync_all();
    if (rank == 0 && threadIdx.x == 0) {
      cg::cluster_group cl = cg::this_cluster();
      x = 0.f;
      y = 0.f;
#pragma unroll
      for (int r = 0; r < C; ++r) {
        const float2 w = *cl.map_shared_rank(part, r);
        x += w.x;
        y += w.y;
      }
    }
  }
}

// Every CTA folds the step-2 partials of the C CTAs in rank order (all end
// with identical sums; used when every CTA needs sigma).
template <int C>
__device__ __forceinline__ void cluster_sum2_all(float& x, float& y, float2* part) {
  if constexpr (C > 1) {
    if (threadIdx.x == 0) *part = make_float2(x, y);
    cluster_sync_all();
    cg::cluster_group cl = cg::this_cluster();
    x = 0.f;
    y = 0.f;
#pragma unroll
    for (int r = 0; r < C; ++r) {
      const float2 w = *cl.map_shared_rank(part, r);
      x += w.x;
      y += w.y;
    }
  }
}

// Bulk prefetch of [p, p + bytes) into L2 with a cache policy (one TMA
// request; p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes, uint64_t pol) {
  asm volatile(
      "{\n\t.reg .u64 g;\n\tcvta.to.global.u64 g, %0;\n\t"
      "cp.async.bulk.prefetch.L2.global.L2::cache_hint [g], %1, %2;\n\t}" ::"l"(p),
      "r"(bytes), "l"(pol)
      : "memory");
}

// Cross-entropy alone streams each row once: thread 0 requests the CTA's
// slice kPrefetchSteps steps ahead of the ring into L2, so HBM sees more
// bytes in flight than the ring holds.  (The fused passes keep rows in L2
// for later passes; there, extra prefetched bytes evict rows still needed,
// measured slower.)
constexpr int kPrefetchSteps = 6;

// One element pair of step 2: sig_p += p*sign(p - q), sig_q += q*sign(p - q).
__device__ __forceinline__ void tvd_accum1(float xs, float xt, float ns2, float nt2,
                                           float& sig_p, float& sig_q) {
  const float p = ex2(fmaf(xs, kLog2e, ns2));
  const float q = ex2(fmaf(xt, kLog2e, nt2));
  const float sg = sgn_pq(p, q);
  sig_p = fmaf(p, sg, sig_p);
  sig_q = fmaf(q, sg, sig_q);
}

template <bool kTvd>
__device__ __forceinline__ void write_row(const FwdArgs& p, int64_t row, int64_t tg, float lse_s,
                                          float lse_t, float abs_sum, float sig, float s_at_tg) {
  p.lse_s[row] = lse_s;
  if constexpr (kTvd) {
    p.tvd[row] = 0.5f * abs_sum;
    p.lse_t[row] = lse_t;
    p.sigma[row] = sig;
  }
  if (tg < 0 || tg >= p.V) {
    p.ce[row] = __uint_as_float(0x7fc00000u);
    if (p.dev_status) atomicOr(p.dev_status, FCT_DEV_TARGET_OUT_OF_RANGE);
  } else {
    p.ce[row] = lse_s - s_at_tg;
  }
}

template <bool kTvd>
__device__ __forceinline__ void write_ignored(const FwdArgs& p, int64_t row) {
  p.ce[row] = 0.f;
  p.lse_s[row] = 0.f;
  if constexpr (kTvd) {
    p.tvd[row] = 0.f;
    p.lse_t[row] = 0.f;
    p.sigma[row] = 0.f;
  }
}

// ===================================================================== pipelined path
//
// Per thread, the sequence of steps is: for each non-ignored row of this
// cluster (rows cluster_id, cluster_id + n_clusters, ...), step 1's n_my
// vectors, then (fused loss only) step 2's n_my vectors, then (single launch)
// step 3's, kPerStep vectors per tensor (NT vectors apart) per step.  Both
// the feed and the consumer walk this same sequence; the feed runs
// kStages - 1 steps ahead of the step being read.

constexpr int kPerStep = 4;  // vectors per tensor moved by one step

// A step's vector count known at compile time (full steps).
template <int N>
struct Count {
  __device__ __forceinline__ constexpr operator int() const { return N; }
};
constexpr int kStages = 3;   // ring slots per thread: two steps in flight while one is read
// Single launch: step 2 leaves one sign bit per element in shared memory, one
// 32-bit word per step of a row, so step 3 needs the student row only (and
// the teacher row may leave L2 after step 2).  Up to kMaxSignWords steps per
// row per thread (V <= 262,144 bf16 with one CTA of 512 threads per row);
// beyond that step 3 re-reads the teacher as well.
constexpr int kMaxSignWords = 16;

// Interleaved start groups of the clusters of a multi-pass launch.
constexpr int kStaggerGroups = 8;

// The feed: this thread's cursor in the sequence, issuing one step of
// cp.async copies per call.  A pass of a row is n_full full steps of
// kPerStep vectors and, if rem > 0, one final step of rem vectors.
template <typename T, int VE, bool kTvd, bool kGrad, int NT>
struct Feed {
  static constexpr int kPasses = kTvd ? (kGrad ? 3 : 2) : (kGrad ? 2 : 1);
  static constexpr int kTensors = kTvd ? 2 : 1;
  static constexpr uint32_t kSlotBytes = kTensors * kPerStep * NT * 16;
  static constexpr int64_t kStride = int64_t(NT) * 16;  // bytes between a thread's vectors

  const char* sp;  // student bytes of the current step's first vector
  const char* tp;  // teacher bytes of the current step's first vector
  int64_t row;
  int32_t q;       // step within the pass
  int32_t pass;
  int32_t n_full, rem;
  int32_t passes_t;  // passes that read the teacher (2 when step 3 uses sign bits)
  bool active;     // false once this thread's sequence is exhausted
  int64_t first_byte;  // byte offset of this thread's first vector within a row
  uint32_t ring;       // shared address of this thread's 16 bytes in slot 0
  uint64_t keep, drop, pol_s, pol_t;

  __device__ __forceinline__ void seek_row(const FwdArgs& p) {
    sp = static_cast<const char*>(p.student) + (row * p.ld_s) * int64_t(sizeof(T)) + first_byte;
    if constexpr (kTvd)
      tp = static_cast<const char*>(p.teacher) + (row * p.ld_t) * int64_t(sizeof(T)) + first_byte;
    // keep each row in L2 until its last pass reads it
    pol_s = (pass + 1 < kPasses) ? keep : drop;
    pol_t = (pass + 1 < passes_t) ? keep : drop;
  }

  __device__ __forceinline__ void next_row(const FwdArgs& p, int64_t n_clusters) {
    row += n_clusters;
    while (row < p.BT && p.target[row] == p.ignore_index) row += n_clusters;
    active = row < p.BT;
    if (active) seek_row(p);
  }

  template <int kCount>
  __device__ __forceinline__ void copy(uint32_t dst, int count) {
    if constexpr (kCount == 4 && kPerStep == 4) {  // a full step: offsets folded
      cp_async16x4<0, NT * 16, static_cast<int>(kStride)>(dst, sp, pol_s);
      if constexpr (kTvd) {
        if (!kGrad || pass < passes_t)
          cp_async16x4<kPerStep * NT * 16, NT * 16, static_cast<int>(kStride)>(dst, tp, pol_t);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kPerStep; ++u) {
        if (kCount == kPerStep || u < count) {
          cp_async16(dst + u * NT * 16, sp + u * kStride, pol_s);
          if constexpr (kTvd) {
            if (!kGrad || pass < passes_t)
              cp_async16(dst + (kPerStep + u) * NT * 16, tp + u * kStride, pol_t);
          }
        }
      }
    }
  }

  // Issue the next step's copies into `slot` and commit one group (an empty
  // group once the sequence is exhausted, so group counting stays uniform).
  __device__ __forceinline__ void feed(const FwdArgs& p, int slot, int64_t n_clusters) {
    if (active) {
      const uint32_t dst = ring + slot * kSlotBytes;
      if (q < n_full) {
        copy<kPerStep>(dst, kPerStep);
      } else {
        copy<0>(dst, rem);
      }
      sp += kPerStep * kStride;
      if constexpr (kTvd) tp += kPerStep * kStride;
      if (++q == n_full + (rem ? 1 : 0)) {
        q = 0;
        if (++pass == kPasses) {
          pass = 0;
          next_row(p, n_clusters);
        } else {
          seek_row(p);
        }
      }
    }
    cp_async_commit();
  }
};

// One pass of the consumer over this thread's vectors of the current row,
// one step at a time: fn(cell, n, k0) with the step's n vectors at
// cell[u*NT] (student) and cell[(kPerStep + u)*NT] (teacher), u < n, being
// this thread's vectors k0 .. k0+n-1.  n is a compile-time constant for full
// steps.  Each slot is refilled with the feed's next step once read.
template <int NT, int kTensors, class FeedT, class Fn>
__device__ __forceinline__ void consume_pass(FeedT& f, int& slot, const FwdArgs& p,
                                             int64_t n_clusters, const uint4* mine, int n_full,
                                             int rem, Fn&& fn) {
  constexpr int kSlotVecs = kTensors * kPerStep * NT;
  for (int q = 0; q < n_full; ++q) {
    cp_async_wait<kStages - 1>();
    fn(mine + slot * kSlotVecs, Count<kPerStep>{}, q * kPerStep);
    f.feed(p, slot, n_clusters);
    slot = (slot + 1 == kStages) ? 0 : slot + 1;
  }
  if (rem) {
    cp_async_wait<kStages - 1>();
    fn(mine + slot * kSlotVecs, rem, n_full * kPerStep);
    f.feed(p, slot, n_clusters);
    slot = (slot + 1 == kStages) ? 0 : slot + 1;
  }
}

// Step-1 update with one step's vectors of one tensor.  The exponents are
// taken against the running reference st.m2 without a per-vector maximum;
// only when the step's sum reaches 2^64 (or is not finite: the first step of
// a row, a new maximum far above the old one, non-finite data) is the step
// redone against its own maximum.  Values up to 2^64 above the reference
// stay exact in fp32 and the sums cannot overflow (2^64 * 2^31 < 2^128).
template <typename T, int VE, int NT, class N>
__device__ __forceinline__ void lse_step(Lse2x& st, const uint4* cell, N n) {
  // two accumulation chains, advanced together by packed (f32x2) adds; the
  // exponent arguments of neighbouring elements by packed FMAs
  float2 acc = make_float2(0.f, 0.f);
  auto sum_exp = [&](float nm) {
    acc = make_float2(0.f, 0.f);
    const float2 L2 = make_float2(kLog2e, kLog2e), nm2 = make_float2(nm, nm);
#pragma unroll
    for (int u = 0; u < kPerStep; ++u) {
      if (u < int(n)) {
        float x[VE];
        unpack_raw<T, VE>(cell[u * NT], x);
#pragma unroll
        for (int j = 0; j < VE; j += 2) {
          const float2 e = __ffma2_rn(make_float2(x[j], x[j + 1]), L2, nm2);
          acc = __fadd2_rn(acc, make_float2(ex2(e.x), ex2(e.y)));
        }
      }
    }
  };
  sum_exp(-st.m2);
  if (!(acc.x + acc.y < 0x1p64f)) {
    float vm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kPerStep; ++u) {
      if (u < int(n)) {
        float x[VE];
        unpack_raw<T, VE>(cell[u * NT], x);
        vm = fmaxf(vm, vec_max(x));
      }
    }
    const float m2n = vm * kLog2e;
    if (m2n > st.m2) {
      const float sc = ex2(st.m2 - m2n);
      st.s.x *= sc;
      st.s.y *= sc;
      st.m2 = m2n;
    }
    if (st.m2 == -INFINITY) {  // every value so far is -inf: nothing to add
      acc = make_float2(0.f, 0.f);
    } else {
      sum_exp(-st.m2);
    }
  }
  st.s = __fadd2_rn(st.s, acc);
}

// lse_step on a step's vectors given by an accessor, cell(u) for u < n (the
// same arithmetic and order as lse_step).
template <typename T, int VE, class Get, class N>
__device__ __forceinline__ void lse_step_get(Lse2x& st, Get&& cell, N n) {
  float2 acc = make_float2(0.f, 0.f);
  auto sum_exp = [&](float nm) {
    acc = make_float2(0.f, 0.f);
    const float2 L2 = make_float2(kLog2e, kLog2e), nm2 = make_float2(nm, nm);
#pragma unroll
    for (int u = 0; u < kPerStep; ++u) {
      if (u < int(n)) {
        float x[VE];
        unpack_raw<T, VE>(cell(u), x);
#pragma unroll
        for (int j = 0; j < VE; j += 2) {
          const float2 e = __ffma2_rn(make_float2(x[j], x[j + 1]), L2, nm2);
          acc = __fadd2_rn(acc, make_float2(ex2(e.x), ex2(e.y)));
        }
      }
    }
  };
  sum_exp(-st.m2);
  if (!(acc.x + acc.y < 0x1p64f)) {
    float vm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kPerStep; ++u) {
      if (u < int(n)) {
        float x[VE];
        unpack_raw<T, VE>(cell(u), x);
        vm = fmaxf(vm, vec_max(x));
      }
    }
    const float m2n = vm * kLog2e;
    if (m2n > st.m2) {
      const float sc = ex2(st.m2 - m2n);
      st.s.x *= sc;
      st.s.y *= sc;
      st.m2 = m2n;
    }
    if (st.m2 == -INFINITY) {  // every value so far is -inf: nothing to add
      acc = make_float2(0.f, 0.f);
    } else {
      sum_exp(-st.m2);
    }
  }
  st.s = __fadd2_rn(st.s, acc);
}

// TG: element type of the gradient written by the single launch (the logits'
// type, or bf16 for fp32 logits).  kSigns: the forward alone also stores each
// element's sign bit and a per-row tie flag for the backward (sign words).
template <typename T, int VE, int C, bool kTvd, bool kGrad, int NT, typename TG = T,
          bool kSigns = false>
__global__ void __launch_bounds__(NT, 1) forward_pipelined(FwdArgs p) {
  static_assert(!kSigns || (kTvd && !kGrad), "sign words come from the forward alone");
  constexpr bool kBits = kGrad || kSigns;  // step 2 builds sign words
  using F = Feed<T, VE, kTvd, kGrad, NT>;
  extern __shared__ __align__(16) uint4 ring_mem[];
  __shared__ float4 red_lse[kMaxWarps];
  __shared__ float2 red_sum[kMaxWarps];
  __shared__ float4 part_lse;
  __shared__ float2 part_sum;

  const int rank = (C > 1) ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
  const int64_t cluster_id = blockIdx.x / C;
  const int64_t n_clusters = gridDim.x / C;
  const int64_t nvec = p.V / VE;
  const int64_t tail0 = nvec * VE;
  const int64_t per = (nvec + C - 1) / C;
  const int64_t vb = min(nvec, rank * per);
  const int64_t ve = min(nvec, vb + per);
  const int64_t span = ve - vb;
  const int tid = threadIdx.x;
  const bool owns_tail = (rank == C - 1);

  // this thread's vectors in each pass of a row: vb + tid + k*NT, k < n_my
  const int n_my = (span > tid) ? static_cast<int>((span - tid + NT - 1) / NT) : 0;
  const int n_full = n_my / kPerStep, rem = n_my % kPerStep;

  F f;
  f.n_full = n_full;
  f.rem = rem;
  f.first_byte = (vb + tid) * 16;
  f.ring = static_cast<uint32_t>(__cvta_generic_to_shared(ring_mem)) + tid * 16;
  f.keep = p.keep_normal ? policy_evict_normal() : policy_evict_last();
  f.drop = policy_evict_first();
  f.q = 0;
  f.pass = 0;
  // steps per row of the thread with the most vectors (thread 0)
  const int64_t max_steps = ((span + NT - 1) / NT + kPerStep - 1) / kPerStep;
  const bool use_bits = kGrad && kTvd && max_steps <= kMaxSignWords;
  f.passes_t = use_bits ? 2 : F::kPasses;
  f.row = cluster_id;
  while (f.row < p.BT && p.target[f.row] == p.ignore_index) f.row += n_clusters;
  f.active = (n_my > 0) && (f.row < p.BT);
  if (f.active) f.seek_row(p);

  // this thread's 16-byte cells: ring_mem[((slot*kTensors + tensor)*kPerStep + u)*NT + tid]
  const uint4* mine = ring_mem + tid;
  // sign words of step 2 after the ring: word w of this thread at sbits[w*NT + tid]
  uint32_t* sbits = reinterpret_cast<uint32_t*>(ring_mem + kStages * F::kTensors * kPerStep * NT);
  // Clusters start staggered in kStaggerGroups interleaved groups: started
  // together, every SM runs its HBM-bound first pass at the same moment and
  // its L2-bound later passes at the same moment, and they stay roughly in
  // step.  Consecutive clusters go to different groups, so each group is
  // spread over the whole chip.  The wait is bounded by the clock and by an
  // iteration count.
  if (p.stagger > 0) {
    const long long wait =
        static_cast<long long>(p.stagger * (cluster_id % kStaggerGroups) / kStaggerGroups);
    const long long t0 = clock64();
    for (int it = 0; it < (1 << 22) && clock64() - t0 < wait; ++it) {
    }
  }
#pragma unroll
  for (int s = 0; s < kStages; ++s) f.feed(p, s, n_clusters);
  int slot = 0;

  const T* S = static_cast<const T*>(p.student);
  const T* Tt = static_cast<const T*>(p.teacher);

  for (int64_t row = cluster_id; row < p.BT; row += n_clusters) {
    const int64_t tg = p.target[row];
    if (tg == p.ignore_index) {
      if (rank == 0 && tid == 0) write_ignored<kTvd>(p, row);
      if constexpr (kGrad) {  // this CTA's slice of the gradient row is zero
        TG* grow = static_cast<TG*>(p.grad) + row * p.ld_g;
        const float zero[VE] = {};
        for (int64_t v = vb + tid; v < ve; v += NT)
          store_grad<T, TG, VE>(grow + v * VE, zero, f.drop);
        if (owns_tail && tail0 + tid < p.V) Elem<TG>::store1(grow + tail0 + tid, 0.f);
      }
      continue;  // uniform over the cluster; the feed skips this row too
    }
    const T* srow = S + row * p.ld_s;
    const T* trow = kTvd ? Tt + row * p.ld_t : nullptr;
    // The row's tie flag starts clear; threads that meet a tie set it after
    // step 2 (past the CTA / cluster barriers that follow this store).
    uint32_t* tie_flag = nullptr;
    if constexpr (kSigns) {
      tie_flag = reinterpret_cast<uint32_t*>(p.signs + row * p.ld_signs);
      if (rank == 0 && tid == 0) *tie_flag = 0u;
    }
    // Read before any gradient of this row can overwrite it (in place).
    const float s_tg =
        (rank == 0 && tid == 0 && tg >= 0 && tg < p.V) ? Elem<T>::load1(srow + tg) : 0.f;
    // ---- step 1: log-sum-exp of both rows
    Lse2x a = lse2x_empty(), b = lse2x_empty();
    consume_pass<NT, F::kTensors>(f, slot, p, n_clusters, mine, n_full, rem,
                                  [&](const uint4* cell, auto n, int k0) {
                                    if constexpr (!kTvd) {
                                      constexpr int64_t kChunk = int64_t(kPerStep) * NT * 16;
                                      const int64_t off = (k0 / kPerStep + kPrefetchSteps) * kChunk;
                                      if (tid == 0 && off < span * 16)
                                        prefetch_l2(reinterpret_cast<const char*>(srow) + vb * 16 + off,
                                                    static_cast<uint32_t>(min(kChunk, span * 16 - off)),
                                                    f.pol_s);
                                    }
                                    lse_step<T, VE, NT>(a, cell, n);
                                    if constexpr (kTvd) lse_step<T, VE, NT>(b, cell + kPerStep * NT, n);
                                  });
    Lse2 fa = lse2x_fold(a), fb = lse2x_fold(b);
    if (owns_tail && tail0 + tid < p.V) {
      float xs[1] = {Elem<T>::load1(srow + tail0 + tid)};
      lse2_update(fa, xs);
      if constexpr (kTvd) {
        float xt[1] = {Elem<T>::load1(trow + tail0 + tid)};
        lse2_update(fb, xt);
      }
    }
    block_merge2<NT>(fa, fb, red_lse);
    cluster_merge2<C>(fa, fb, &part_lse);
    const float lse_s = lse2_finish(fa);

    if constexpr (!kTvd) {
      if (rank == 0 && tid == 0) write_row<false>(p, row, tg, lse_s, 0.f, 0.f, 0.f, s_tg);
      // peers may still read part_lse; warps may still read red_lse
      if constexpr (C > 1) {
        cluster_sync_all();
      } else {
        __syncthreads();
      }
      if constexpr (kGrad) {
        // ---- cross-entropy alone in one launch: a second pass over the
        // L2-resident row writes grad_ce * (p - [v == target]) with the
        // backward kernel's expressions, so the result is bit-identical.
        const float gce = p.grad_ce[row * p.grad_stride];
        const float ns2 = -(lse_s * kLog2e);
        const bool bad = (tg < 0 || tg >= p.V);
        TG* grow = static_cast<TG*>(p.grad) + row * p.ld_g;
        TG* gmine = grow + (vb + tid) * VE;
        const int64_t tg_rel = tg - (vb + tid) * VE;
        const float2 L2 = make_float2(kLog2e, kLog2e), ns22 = make_float2(ns2, ns2);
        consume_pass<NT, F::kTensors>(
            f, slot, p, n_clusters, mine, n_full, rem, [&](const uint4* cell, auto n, int k0) {
#pragma unroll
              for (int u = 0; u < kPerStep; ++u) {
                if (u < int(n)) {
                  float xs[VE], g[VE];
                  unpack_raw<T, VE>(cell[u * NT], xs);
#pragma unroll
                  for (int j = 0; j < VE; j += 2) {
                    const float2 e = __ffma2_rn(make_float2(xs[j], xs[j + 1]), L2, ns22);
                    g[j] = ex2(e.x) * gce;
                    g[j + 1] = ex2(e.y) * gce;
                  }
                  const int64_t off = tg_rel - int64_t(k0 + u) * NT * VE;
                  if (static_cast<uint64_t>(off) < static_cast<uint64_t>(VE)) {
#pragma unroll
                    for (int j = 0; j < VE; ++j)
                      if (j == off) g[j] -= gce;
                  }
                  if (bad) {
#pragma unroll
                    for (int j = 0; j < VE; ++j) g[j] = __uint_as_float(0x7fc00000u);
                  }
                  store_grad<T, TG, VE>(gmine + int64_t(k0 + u) * NT * VE, g, f.drop);
                }
              }
            });
        if (owns_tail && tail0 + tid < p.V) {
          const int64_t v = tail0 + tid;
          float g = ex2(fmaf(Elem<T>::load1(srow + v), kLog2e, ns2)) * gce;
          if (v == tg) g -= gce;
          Elem<TG>::store1(grow + v, bad ? __uint_as_float(0x7fc00000u) : g);
        }
      }
    } else {
      const float lse_t = lse2_finish(fb);
      // The backward recomputes p and q from the stored lse values with this
      // same expression (x*log2e - lse*log2e, one FMA, then ex2), so both
      // kernels see bit-identical p and q.
      const float ns2 = -(lse_s * kLog2e);
      const float nt2 = -(lse_t * kLog2e);

      // ---- step 2: sigma = sum p*sign(p - q) and tau = sum q*sign(p - q);
      // sum |p - q| = sigma - tau.  Ties have sign 0 and add nothing.
      float sig_p = 0.f, sig_q = 0.f;
      const float2 L2 = make_float2(kLog2e, kLog2e), nst = make_float2(ns2, nt2);
      auto tvd_pair = [&](float xs, float xt) {  // one element (the row's ragged tail)
        // the student and teacher exponents of one element in one packed FMA
        // (each lane rounds exactly like the scalar fmaf of the backward)
        const float2 e = __ffma2_rn(make_float2(xs, xt), L2, nst);
        const float pp = ex2(e.x);
        const float qq = ex2(e.y);
        const float sg = sgn_pq(pp, qq);
        sig_p = fmaf(pp, sg, sig_p);
        sig_q = fmaf(qq, sg, sig_q);
      };
      // Two neighbouring elements at a time, each tensor's pair in one packed
      // op (neighbours of one tensor come out of the unpack side by side);
      // sigma and tau run as two packed partial sums.
      const float2 ns22 = make_float2(ns2, ns2), nt22 = make_float2(nt2, nt2);
      float2 sp2 = make_float2(0.f, 0.f), sq2 = make_float2(0.f, 0.f);
      auto tvd_two = [&](float s0, float s1, float t0, float t1) {
        const float2 es = __ffma2_rn(make_float2(s0, s1), L2, ns22);
        const float2 et = __ffma2_rn(make_float2(t0, t1), L2, nt22);
        const float2 pp = make_float2(ex2(es.x), ex2(es.y));
        const float2 qq = make_float2(ex2(et.x), ex2(et.y));
        const float2 sg = sgn_pq2(pp, qq);
        sp2 = __ffma2_rn(pp, sg, sp2);
        sq2 = __ffma2_rn(qq, sg, sq2);
        return sg;
      };
      // Single launch: the sign bit of each element (1 for p < q), shifted in
      // element order into one word per step, and the AND of all signs' bit
      // patterns, whose exponent bits clear at a tie (sign +0) and at a
      // subnormal difference (a sign strictly between -1 and 1).
      uint32_t tie_and = 0xffffffffu;
      consume_pass<NT, F::kTensors>(f, slot, p, n_clusters, mine, n_full, rem,
                                    [&](const uint4* cell, auto n, int k0) {
                                      [[maybe_unused]] uint32_t word = 0;
#pragma unroll
                                      for (int u = 0; u < kPerStep; ++u) {
                                        if (u < int(n)) {
                                          float xs[VE], xt[VE];
                                          unpack_raw<T, VE>(cell[u * NT], xs);
                                          unpack_raw<T, VE>(cell[(kPerStep + u) * NT], xt);
#pragma unroll
                                          for (int j = 0; j < VE; j += 2) {
                                            const float2 sg = tvd_two(xs[j], xs[j + 1], xt[j], xt[j + 1]);
                                            if constexpr (kBits) {
                                              const uint32_t b0 = __float_as_uint(sg.x);
                                              const uint32_t b1 = __float_as_uint(sg.y);
                                              word = __funnelshift_l(b1, __funnelshift_l(b0, word, 1), 1);
                                              tie_and &= b0 & b1;
                                            }
                                          }
                                        }
                                      }
                                      if constexpr (kBits) {
                                        // a short step's bits move up to the full step's positions
                                        if (int(n) < kPerStep) word <<= (kPerStep - int(n)) * VE;
                                      }
                                      if constexpr (kGrad) {
                                        if (use_bits) sbits[(k0 / kPerStep) * NT + tid] = word;
                                      }
                                      if constexpr (kSigns) {
                                        // one byte per vector: its VE bits, element j at bit VE-1-j
                                        uint8_t* dst = p.signs + row * p.ld_signs + 4 + vb + tid +
                                                       int64_t(k0) * NT;
#pragma unroll
                                        for (int u = 0; u < kPerStep; ++u)
                                          if (u < int(n))
                                            dst[u * NT] = static_cast<uint8_t>(
                                                (word >> (kPerStep * VE - VE * (u + 1))) &
                                                ((1u << VE) - 1u));
                                      }
                                    });
      if constexpr (kSigns) {
        if ((tie_and & 0x3f800000u) != 0x3f800000u) atomicOr(tie_flag, 1u);
      }
      sig_p = sp2.x + sp2.y;
      sig_q = sq2.x + sq2.y;
      if (owns_tail && tail0 + tid < p.V)
        tvd_pair(Elem<T>::load1(srow + tail0 + tid), Elem<T>::load1(trow + tail0 + tid));
      float abs_sum = sig_p - sig_q;
      float sig = sig_p;
      block_sum2<NT>(abs_sum, sig, red_sum);
      if constexpr (kGrad) {
        cluster_sum2_all<C>(abs_sum, sig, &part_sum);
      } else {
        cluster_sum2<C>(abs_sum, sig, &part_sum, rank);
      }
      if (rank == 0 && tid == 0) write_row<true>(p, row, tg, lse_s, lse_t, abs_sum, sig, s_tg);

      if constexpr (kGrad) {
        // ---- step 3: the "Backward Pass" gradient, same expressions as the
        // backward kernel: grad = p * c(sign) - grad_ce * [v == target].
        const float gce = p.grad_ce[row * p.grad_stride];
        const float h = 0.5f * p.grad_tvd[row * p.grad_stride];
        const float c0 = gce - h * sig;  // coefficient of p: c0 + h * sign
        const bool bad = (tg < 0 || tg >= p.V);
        TG* grow = static_cast<TG*>(p.grad) + row * p.ld_g;
        TG* gmine = grow + (vb + tid) * VE;
        // element offset of the target from this thread's first element
        const int64_t tg_rel = tg - (vb + tid) * VE;
        auto grad_of = [&](float xs, float xt) {
          const float2 e = __ffma2_rn(make_float2(xs, xt), L2, nst);
          const float pp = ex2(e.x);
          return pp * fmaf(h, sgn_pq(pp, ex2(e.y)), c0);
        };
        auto finish_vec = [&](float (&g)[VE], int k) {
          const int64_t off = tg_rel - int64_t(k) * NT * VE;
          if (static_cast<uint64_t>(off) < static_cast<uint64_t>(VE)) {
#pragma unroll
            for (int j = 0; j < VE; ++j)
              if (j == off) g[j] -= gce;
          }
          if (bad) {
#pragma unroll
            for (int j = 0; j < VE; ++j) g[j] = __uint_as_float(0x7fc00000u);
          }
          store_grad<T, TG, VE>(gmine + int64_t(k) * NT * VE, g, f.drop);
        };
        auto grad_vec = [&](const uint4 ws, const uint4 wt, int k) {
          float xs[VE], xt[VE], g[VE];
          unpack_raw<T, VE>(ws, xs);
          unpack_raw<T, VE>(wt, xt);
#pragma unroll
          for (int j = 0; j < VE; ++j) g[j] = grad_of(xs[j], xt[j]);
          finish_vec(g, k);
        };
        // With step 2's sign bits and no tie in this thread's elements, the
        // coefficient of p is one of fmaf(h, +-1, c0), the values the backward
        // kernel's expression takes at sign +-1, so the gradient is bit-identical.
        const bool from_bits = use_bits && (tie_and & 0x3f800000u) == 0x3f800000u;
        const float c_plus = fmaf(h, 1.f, c0), c_minus = fmaf(h, -1.f, c0);
        const float2 ns22 = make_float2(ns2, ns2);
        const T* tmine = trow + (vb + tid) * VE;
        consume_pass<NT, F::kTensors>(
            f, slot, p, n_clusters, mine, n_full, rem, [&](const uint4* cell, auto n, int k0) {
              if (from_bits) {
                const uint32_t word = sbits[(k0 / kPerStep) * NT + tid];
#pragma unroll
                for (int u = 0; u < kPerStep; ++u) {
                  if (u < int(n)) {
                    float xs[VE], g[VE];
                    unpack_raw<T, VE>(cell[u * NT], xs);
#pragma unroll
                    for (int j = 0; j < VE; j += 2) {
                      const float2 e = __ffma2_rn(make_float2(xs[j], xs[j + 1]), L2, ns22);
                      constexpr int kBits = kPerStep * VE;
                      const int b0 = kBits - 1 - (u * VE + j);
                      const float ca = ((word >> b0) & 1u) ? c_minus : c_plus;
                      const float cb = ((word >> (b0 - 1)) & 1u) ? c_minus : c_plus;
                      const float2 gg = __fmul2_rn(make_float2(ex2(e.x), ex2(e.y)),
                                                   make_float2(ca, cb));
                      g[j] = gg.x;
                      g[j + 1] = gg.y;
                    }
                    finish_vec(g, k0 + u);
                  }
                }
              } else {
#pragma unroll
                for (int u = 0; u < kPerStep; ++u) {
                  if (u < int(n)) {
                    // the teacher comes from the ring unless step 3 was planned
                    // on sign bits (then it was not copied: read it from L2/HBM)
                    const uint4 wt =
                        use_bits ? load_raw<T, VE>(tmine + int64_t(k0 + u) * NT * VE, f.drop)
                                 : cell[(kPerStep + u) * NT];
                    grad_vec(cell[u * NT], wt, k0 + u);
                  }
                }
              }
            });
        if (owns_tail && tail0 + tid < p.V) {
          const int64_t v = tail0 + tid;
          float g = grad_of(Elem<T>::load1(srow + v), Elem<T>::load1(trow + v));
          if (v == tg) g -= gce;
          Elem<TG>::store1(grow + v, bad ? __uint_as_float(0x7fc00000u) : g);
        }
      }
    }
  }
  cp_async_wait_all();
  // No CTA may leave while a peer can still read its shared memory.
  if constexpr (C > 1) cluster_sync_all();
}

// ===================================================================== bulk-copy (TMA) ring path
//
// The same three passes with a CTA-wide ring filled by the TMA unit: one
// producer lane issues, per step, one cp.async.bulk per tensor (the step's
// kPerStep * NT contiguous 16-byte vectors, 32 KB) into a ring slot and
// arms the slot's "full" mbarrier with the byte count; the NT consumer
// threads wait on it, read their cells exactly where the per-thread ring
// puts them (vector u*NT + tid of the step), and each consumer warp arrives
// on the slot's "empty" mbarrier when done, which lets the producer refill
// it.  The consumers issue no copy instructions and keep no feed state.  A
// row belongs to one CTA (no cluster).  The arithmetic is that of
// forward_pipelined with one CTA per row; step 1 folds its partial sums once
// per step of kPS vectors, so the per-row outputs equal forward_pipelined's
// to rounding (bit for bit when kPS == kPerStep), and the forward alone and
// the single launch of this ring agree bit for bit with each other (the
// backward reads only their per-row outputs).  In step 3 the target
// element's gradient is written by the
// thread that owns it after its vector stores (same thread, same address,
// so the later store wins), which takes the target test out of the
// per-vector loop.
//
// Every mbarrier wait is bounded (about 2 s of clock): a wait that runs out
// sets a CTA-wide abort flag, after which every wait returns at once, the
// producer stops issuing, and the kernel ORs FCT_DEV_WAIT_TIMEOUT into the
// status word (the outputs are then invalid).

// Bulk copy of `bytes` (a multiple of 16) from global `src` into this CTA's
// shared memory at `dst` (both 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t pol) {
  asm volatile(
      "{\n\t.reg .u64 g;\n\tcvta.to.global.u64 g, %1;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [g], %2, [%3], %4;\n\t}" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// Which steps each pass of a row stages in the ring, shared by the producer
// and the consumers.  The passes by role: 0 = step 1 (log-sum-exp; absent
// when the states are given), 1 = step 2 (sums and sign bits), 2 = step 3
// (gradient).  Each pass stages its steps in increasing order, except:
// * c1: step 1's last c1 steps stay in their slots; step 2 computes them
//   first and stages only [0, n - c1).
// * c3: step 2's last c3 staged steps [a3, a3 + c3), a3 = n - c1 - c3, stay
//   in the slots' student halves; step 3 (student only, on sign bits)
//   computes them first and stages its other steps into the teacher halves.
// Each carried step is read from L2 once less per row.
struct RingPlan {
  int n;          // steps per pass
  int c1, c3;     // steps carried from step 1 to 2, from step 2 to 3
  bool teacher3;  // step 3 stages the teacher (no sign bits)
  __device__ int a3() const { return n - c1 - c3; }
  __device__ bool staged3(int q) const { return q < a3() || q >= n - c1; }
};

// The producer lane: walks the consumers' sequence (rows of this CTA that
// are not ignored; per row the passes of kRole0..kRoles-1, each staging the
// steps RingPlan gives) and fills ring slot t % kST for fill t.  In the first
// pass (from HBM) it also asks L2 for the chunks kPref steps ahead, so more
// of the row is on its way than the ring holds.  Each tensor's step is read
// with evict_last (or evict_normal) while a later pass of the row stages it
// again, else with evict_first.  With c3 > 0 a row's first fill also waits
// until the consumers have computed the previous row's steps carried into
// its step 3 (carry_bar): those sit in the student halves the fill would
// overwrite.
template <int NT, int kPS, int kST, int kPref, int kRole0, int kRoles, typename T>
__device__ void tma_produce(const FwdArgs& p, uint4* ring_mem, uint64_t* full_bar,
                            uint64_t* empty_bar, uint64_t* carry_bar, volatile int* abort,
                            int64_t nvec, RingPlan rp) {
  constexpr int kStepVecs = kPS * NT;
  constexpr uint32_t kTensorBytes = kStepVecs * 16;
  constexpr bool kStep3 = kRoles == 3;
  const uint64_t keep = p.keep_normal ? policy_evict_normal() : policy_evict_last();
  const uint64_t drop = policy_evict_first();
  const uint32_t ring = smem_addr(ring_mem);
  if (p.stagger > 0) {  // interleaved start groups, as in forward_pipelined
    const long long wait =
        static_cast<long long>(p.stagger * (blockIdx.x % kStaggerGroups) / kStaggerGroups);
    const long long t0 = clock64();
    for (int it = 0; it < (1 << 22) && clock64() - t0 < wait; ++it) {
    }
  }
  auto chunk_bytes = [&](int q) {
    const int64_t v0 = int64_t(q) * kStepVecs;
    return static_cast<uint32_t>(((nvec - v0 < kStepVecs) ? nvec - v0 : kStepVecs) * 16);
  };
  uint32_t t = 0, rows_carried = 0;
  bool ok = rp.n > 0;
  for (int64_t row = blockIdx.x; ok && row < p.BT; row += gridDim.x) {
    if (p.target[row] == p.ignore_index) continue;
    if (rows_carried > 0 && !mbar_wait(carry_bar, (rows_carried - 1) & 1, abort)) break;
    const char* srow = static_cast<const char*>(p.student) + row * p.ld_s * int64_t(sizeof(T));
    const char* trow = static_cast<const char*>(p.teacher) + row * p.ld_t * int64_t(sizeof(T));
    if constexpr (kPref > 0) {  // the first chunks of the first pass
      for (int q = 0; q < kPref && q < rp.n; ++q) {
        prefetch_l2(srow + int64_t(q) * kTensorBytes, chunk_bytes(q), keep);
        prefetch_l2(trow + int64_t(q) * kTensorBytes, chunk_bytes(q), keep);
      }
    }
    for (int role = kRole0; ok && role < kRoles; ++role) {
      const bool with_t = role < 2 || rp.teacher3;
      const bool into_t = role == 2 && rp.c3 > 0;  // the student into the teacher halves
      const int q_end = role == 1 ? rp.n - rp.c1 : rp.n;
      for (int q = 0; q < q_end; ++q) {
        if (role == 2 && !rp.staged3(q)) continue;  // carried from step 2
        const uint32_t slot = t % kST, fill = t / kST;
        if (fill > 0 && !mbar_wait(&empty_bar[slot], (fill - 1) & 1, abort)) {
          ok = false;
          break;
        }
        // staged again by a later pass of this row?
        const bool again2 = role == 0 && q < rp.n - rp.c1;
        const bool s_again = again2 || (kStep3 && role < 2 && rp.staged3(q));
        const bool t_again = again2 || (kStep3 && role < 2 && rp.teacher3);
        const int64_t off = int64_t(q) * kTensorBytes;
        const uint32_t bytes = chunk_bytes(q);
        mbar_arrive_expect_tx(&full_bar[slot], with_t ? 2 * bytes : bytes);
        const uint32_t dst = ring + slot * (2 * kTensorBytes) + (into_t ? kTensorBytes : 0);
        bulk_load(dst, srow + off, bytes, &full_bar[slot], s_again ? keep : drop);
        if (with_t) bulk_load(dst + kTensorBytes, trow + off, bytes, &full_bar[slot], t_again ? keep : drop);
        if constexpr (kPref > 0) {
          if (role == kRole0 && q + kPref < rp.n) {
            const int64_t pf = int64_t(q + kPref) * kTensorBytes;
            prefetch_l2(srow + pf, chunk_bytes(q + kPref), keep);
            prefetch_l2(trow + pf, chunk_bytes(q + kPref), keep);
          }
        }
        ++t;
      }
    }
    if (rp.c3 > 0) ++rows_carried;
  }
  // No copy may still be landing when this CTA exits: wait (bounded, even
  // after an abort) for the last fills.
  for (uint32_t i = (t > uint32_t(kST) ? t - kST : 0); i < t; ++i)
    mbar_wait(&full_bar[i % kST], (i / kST) & 1, abort, /*heed_abort=*/false);
}

// kPS: 16-byte vectors per thread per tensor in one step (a step moves
// kPS * NT contiguous vectors of each tensor); kST: ring slots; kPref: L2
// prefetch distance of the first pass, in steps (0 = none).
// kSigns: the forward alone also stores each element's sign bit and a per-row
// tie flag for the backward (sign words, as forward_pipelined does).
// kLseIn: the single launch with step 1's per-row states given as partials
// (FwdArgs::lse_part_s/t): two passes over the row, the first one fed from
// HBM, and the teacher only in the first when step 3 runs on sign bits, so
// L2 holds just the student between the passes.
// kCarry1, kCarry3: steps carried from step 1 into step 2 (RingPlan::c1; at
// most kST - 1, so one slot stays free for step 2's first fill, and only
// with one step per sign word) and from step 2 into step 3 (RingPlan::c3,
// when step 3 runs on sign bits).  Carried steps are computed first in the
// pass they are carried into.  The step order of step 2, and so the rounding
// of its sums, depends only on the row's length, the same in the forward
// alone and in the single launch; step 3's order does not change any value.
template <typename T, int VE, bool kGrad, int NT, typename TG, int kPS, int kST, int kPref,
          bool kSigns = false, bool kLseIn = false, int kCarry1 = 0, int kCarry3 = 0>
__global__ void __launch_bounds__(NT + 32, 1) forward_tma(FwdArgs p) {
  static_assert(kPS >= 1 && kPS <= kPerStep, "steps of at most kPerStep vectors per thread");
  static_assert(!kSigns || !kGrad, "sign words come from the forward alone");
  static_assert(!kLseIn || kGrad, "given log-sum-exp states: the single launch only");
  static_assert(kCarry1 >= 0 && kCarry1 < kST, "a free slot for step 2's first fill");
  static_assert(kCarry3 >= 0 && kCarry3 <= kST, "at most one carried step per slot");
  constexpr bool kWord = kGrad || kSigns;  // step 2 builds sign words
  constexpr int kStepVecs = kPS * NT;       // 16-byte vectors per tensor per step
  constexpr int kSlotVecs = 2 * kStepVecs;  // student then teacher
  // step 2's sign bits: kBits per step, kSpw steps per 32-bit word
  constexpr int kBits = kPS * VE;
  static_assert(32 % kBits == 0, "whole steps per sign word");
  constexpr int kSpw = 32 / kBits;
  // step 2 out of order only where each step has a sign word of its own
  constexpr int kC1 = (kLseIn || kSpw != 1) ? 0 : kCarry1;
  extern __shared__ __align__(128) uint4 bulk_ring[];
  __shared__ __align__(8) uint64_t full_bar[kST];
  __shared__ __align__(8) uint64_t empty_bar[kST];
  __shared__ float4 red_lse[kMaxWarps];
  __shared__ float2 red_sum[kMaxWarps];
  __shared__ __align__(8) uint64_t carry_bar;  // the steps carried into step 3 have been read
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int64_t nvec = p.V / VE;
  const int64_t tail0 = nvec * VE;
  const int n_steps = static_cast<int>((nvec + kStepVecs - 1) / kStepVecs);
  const bool use_bits = kGrad && n_steps <= kMaxSignWords * kSpw;
  RingPlan rp;
  rp.n = n_steps;
  rp.c1 = n_steps >= kC1 + kST ? kC1 : 0;
  rp.c3 = use_bits ? (n_steps - rp.c1 < kCarry3 ? n_steps - rp.c1 : kCarry3) : 0;
  rp.teacher3 = kGrad && !use_bits;

  if (tid == 0) {
    for (int s = 0; s < kST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NT / 32);
    }
    mbar_init(&carry_bar, NT / 32);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();  // the last CTA-wide barrier: from here the producer runs on its own
  if (tid >= NT) {
    if (tid == NT)
      tma_produce<NT, kPS, kST, kPref, kLseIn ? 1 : 0, kGrad ? 3 : 2, T>(
          p, bulk_ring, full_bar, empty_bar, &carry_bar, &abort_flag, nvec, rp);
    return;
  }

  // ---- consumers
  const int lane = tid & 31;
  // this thread's vectors in the last step of a pass (all kPS in the others)
  const int64_t n_last = nvec - int64_t(n_steps > 0 ? n_steps - 1 : 0) * kStepVecs;
  const int64_t cnt_all = (n_last > tid) ? (n_last - tid + NT - 1) / NT : 0;
  const int cnt_last = static_cast<int>(cnt_all < kPS ? cnt_all : kPS);
  const uint4* mine = bulk_ring + tid;
  uint32_t* sbits = reinterpret_cast<uint32_t*>(bulk_ring + kST * kSlotVecs);
  uint32_t slot = 0, parity = 0;  // the next fill's slot and phase
  // fn(cell_s, cell_t, n, q) on step q, with this thread's n vectors of the
  // step as cell_s(u) (student) and cell_t(u) (teacher), u < n
  auto run = [&](const uint4* cells_s, const uint4* cells_t, int q, auto&& fn) {
    auto cs = [&](int u) { return cells_s[u * NT]; };
    auto ct = [&](int u) { return cells_t[u * NT]; };
    if (q + 1 < n_steps || cnt_last == kPS) {
      fn(cs, ct, Count<kPS>{}, q);
    } else {
      fn(cs, ct, cnt_last, q);
    }
  };
  auto arrive = [&](uint64_t* bar) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  // the next fill: wait for it, return its slot, move on
  auto next_fill = [&]() {
    const uint32_t k = slot;
    mbar_wait(&full_bar[k], parity, &abort_flag);
    if (++slot == kST) {
      slot = 0;
      parity ^= 1u;
    }
    return k;
  };
  // slot of the j-th of the last c fills
  auto recent = [&](int c, int j) { return (slot + kST - c + j) % kST; };
  auto cells = [&](uint32_t k) { return mine + k * kSlotVecs; };
  // step 1: every step in order; the last c1 slots are kept for step 2
  auto pass1 = [&](auto&& fn) {
    for (int q = 0; q < n_steps; ++q) {
      const uint32_t k = next_fill();
      run(cells(k), cells(k) + kStepVecs, q, fn);
      if (q < n_steps - rp.c1) arrive(&empty_bar[k]);
    }
  };
  // step 2: step 1's last c1 steps, then the others in order
  auto pass2 = [&](auto&& fn) {
    for (int j = 0; j < rp.c1; ++j) {
      const uint32_t k = recent(rp.c1, j);
      run(cells(k), cells(k) + kStepVecs, n_steps - rp.c1 + j, fn);
      arrive(&empty_bar[k]);
    }
    for (int q = 0; q < n_steps - rp.c1; ++q) {
      const uint32_t k = next_fill();
      run(cells(k), cells(k) + kStepVecs, q, fn);
      arrive(&empty_bar[k]);
    }
  };
  // step 3: with c3 > 0, step 2's last c3 steps from the slots' student
  // halves, then the others from the teacher halves (the teacher is not
  // staged: cell_t is cell_s); else every step in order
  auto pass3 = [&](auto&& fn) {
    if (rp.c3 > 0) {
      for (int j = 0; j < rp.c3; ++j) {
        const uint4* c = cells(recent(rp.c3, j));
        run(c, c, rp.a3() + j, fn);
      }
      arrive(&carry_bar);
      for (int q = 0; q < n_steps; ++q) {
        if (!rp.staged3(q)) continue;
        const uint32_t k = next_fill();
        run(cells(k) + kStepVecs, cells(k) + kStepVecs, q, fn);
        arrive(&empty_bar[k]);
      }
    } else {
      for (int q = 0; q < n_steps; ++q) {
        const uint32_t k = next_fill();
        run(cells(k), cells(k) + kStepVecs, q, fn);
        arrive(&empty_bar[k]);
      }
    }
  };

  const T* S = static_cast<const T*>(p.student);
  const T* Tt = static_cast<const T*>(p.teacher);
  const uint64_t drop = policy_evict_first();
  const float2 L2 = make_float2(kLog2e, kLog2e);

  for (int64_t row = blockIdx.x; row < p.BT; row += gridDim.x) {
    const int64_t tg = p.target[row];
    const T* srow = S + row * p.ld_s;
    const T* trow = Tt + row * p.ld_t;
    if (tg == p.ignore_index) {
      if (tid == 0) write_ignored<true>(p, row);
      if constexpr (kGrad) {  // a zero gradient row
        TG* grow = static_cast<TG*>(p.grad) + row * p.ld_g;
        const float zero[VE] = {};
        for (int64_t v = tid; v < nvec; v += NT) store_grad<T, TG, VE>(grow + v * VE, zero, drop);
        if (tail0 + tid < p.V) Elem<TG>::store1(grow + tail0 + tid, 0.f);
      }
      continue;  // the producer skips this row too
    }
    const bool bad = (tg < 0 || tg >= p.V);
    // Logits read before any gradient of this row can overwrite them (in
    // place): the target logit for ce, and (single launch) the target
    // element's student and teacher logits for the thread that owns it.
    const float s_tg = (tid == 0 && !bad) ? Elem<T>::load1(srow + tg) : 0.f;
    const bool owner = kGrad && !bad && tg < tail0 && ((tg / VE) % NT) == tid;
    // The row's tie flag starts clear; threads that meet a tie set it after
    // step 2 (past the consumers' barrier in step 1's merge).
    uint32_t* tie_flag = nullptr;
    if constexpr (kSigns) {
      tie_flag = reinterpret_cast<uint32_t*>(p.signs + row * p.ld_signs);
      if (tid == 0) *tie_flag = 0u;
    }
    float xs_tg = 0.f, xt_tg = 0.f;
    if (owner) {
      xs_tg = Elem<T>::load1(srow + tg);
      xt_tg = Elem<T>::load1(trow + tg);
    }

    // ---- step 1: log-sum-exp of both rows
    Lse2 fa, fb;
    if constexpr (kLseIn) {
      // the given partial states, thread by thread in index order, then
      // across the threads in the fixed order of block_merge2
      fa = lse2_empty();
      fb = lse2_empty();
      const float2* ps = p.lse_part_s + row * p.lse_ld;
      const float2* pt = p.lse_part_t + row * p.lse_ld;
      for (int64_t j = tid; j < p.lse_n; j += NT) {
        const float2 u = ps[j], w = pt[j];
        fa = lse2_merge(fa, Lse2{u.x, u.y});
        fb = lse2_merge(fb, Lse2{w.x, w.y});
      }
    } else {
      Lse2x a = lse2x_empty(), b = lse2x_empty();
      pass1([&](auto&& cs, auto&& ct, auto n, int) {
        lse_step_get<T, VE>(a, cs, n);
        lse_step_get<T, VE>(b, ct, n);
      });
      fa = lse2x_fold(a);
      fb = lse2x_fold(b);
      if (tail0 + tid < p.V) {
        float xs[1] = {Elem<T>::load1(srow + tail0 + tid)};
        float xt[1] = {Elem<T>::load1(trow + tail0 + tid)};
        lse2_update(fa, xs);
        lse2_update(fb, xt);
      }
    }
    block_merge2<NT, true>(fa, fb, red_lse);
    const float lse_s = lse2_finish(fa);
    const float lse_t = lse2_finish(fb);
    const float ns2 = -(lse_s * kLog2e);
    const float nt2 = -(lse_t * kLog2e);
    const float2 nst = make_float2(ns2, nt2);

    // ---- step 2: sigma and tau (sum |p - q| = sigma - tau), sign bits
    const float2 ns22 = make_float2(ns2, ns2), nt22 = make_float2(nt2, nt2);
    float2 sp2 = make_float2(0.f, 0.f), sq2 = make_float2(0.f, 0.f);
    uint32_t tie_and = 0xffffffffu;
    [[maybe_unused]] uint32_t packed = 0;  // sign bits of the steps of the current word
    pass2([&](auto&& cs, auto&& ct, auto n, int q) {
      [[maybe_unused]] uint32_t word = 0;
#pragma unroll
      for (int u = 0; u < kPS; ++u) {
        if (u < int(n)) {
          float xs[VE], xt[VE];
          unpack_raw<T, VE>(cs(u), xs);
          unpack_raw<T, VE>(ct(u), xt);
#pragma unroll
          for (int j = 0; j < VE; j += 2) {
            const float2 es = __ffma2_rn(make_float2(xs[j], xs[j + 1]), L2, ns22);
            const float2 et = __ffma2_rn(make_float2(xt[j], xt[j + 1]), L2, nt22);
            const float2 pp = make_float2(ex2(es.x), ex2(es.y));
            const float2 qq = make_float2(ex2(et.x), ex2(et.y));
            const float2 sg = sgn_pq2(pp, qq);
            sp2 = __ffma2_rn(pp, sg, sp2);
            sq2 = __ffma2_rn(qq, sg, sq2);
            if constexpr (kWord) {
              const uint32_t b0 = __float_as_uint(sg.x);
              const uint32_t b1 = __float_as_uint(sg.y);
              word = __funnelshift_l(b1, __funnelshift_l(b0, word, 1), 1);
              tie_and &= b0 & b1;
            }
          }
        }
      }
      if constexpr (kWord) {
        // a short step's bits move up to the full step's positions
        if (int(n) < kPS) word <<= (kPS - int(n)) * VE;
      }
      if constexpr (kSigns) {
        // one byte per vector: its VE bits, element j at bit VE-1-j
        uint8_t* dst = p.signs + row * p.ld_signs + 4 + tid + int64_t(q) * kStepVecs;
#pragma unroll
        for (int u = 0; u < kPS; ++u)
          if (u < int(n))
            dst[u * NT] = static_cast<uint8_t>((word >> (kBits - VE * (u + 1))) & ((1u << VE) - 1u));
      }
      if constexpr (kGrad) {
        // the steps of a word go in from the top (first step highest), and a
        // row's last word is shifted as if it were full
        if constexpr (kSpw == 1) {
          packed = word;
        } else {
          packed = (packed << kBits) | word;
        }
        const int i = q % kSpw;
        if (use_bits && (i == kSpw - 1 || q + 1 == n_steps)) {
          if constexpr (kSpw > 1) packed <<= (kSpw - 1 - i) * kBits;
          sbits[(q / kSpw) * NT + tid] = packed;
          packed = 0;
        }
      }
    });
    if constexpr (kSigns) {
      if ((tie_and & 0x3f800000u) != 0x3f800000u) atomicOr(tie_flag, 1u);
    }
    float sig_p = sp2.x + sp2.y;
    float sig_q = sq2.x + sq2.y;
    if (tail0 + tid < p.V) {
      const float2 e = __ffma2_rn(make_float2(Elem<T>::load1(srow + tail0 + tid),
                                              Elem<T>::load1(trow + tail0 + tid)),
                                  L2, nst);
      const float pp = ex2(e.x), qq = ex2(e.y);
      const float sg = sgn_pq(pp, qq);
      sig_p = fmaf(pp, sg, sig_p);
      sig_q = fmaf(qq, sg, sig_q);
    }
    float abs_sum = sig_p - sig_q;
    float sig = sig_p;
    block_sum2<NT, true>(abs_sum, sig, red_sum);
    if (tid == 0) write_row<true>(p, row, tg, lse_s, lse_t, abs_sum, sig, s_tg);

    if constexpr (kGrad) {
      // ---- step 3: grad = p * c(sign) - grad_ce * [v == target], the
      // backward kernel's expressions
      const float gce = p.grad_ce[row * p.grad_stride];
      const float h = 0.5f * p.grad_tvd[row * p.grad_stride];
      const float c0 = gce - h * sig;
      const float c_plus = fmaf(h, 1.f, c0), c_minus = fmaf(h, -1.f, c0);
      TG* grow = static_cast<TG*>(p.grad) + row * p.ld_g;
      TG* gmine = grow + int64_t(tid) * VE;
      const T* tmine = trow + int64_t(tid) * VE;
      const bool from_bits = use_bits && (tie_and & 0x3f800000u) == 0x3f800000u;
      // p * c rounded on its own (never fused with a later subtraction), as
      // the backward kernel's product is
      auto grad_of = [&](float xs, float xt) {
        const float2 e = __ffma2_rn(make_float2(xs, xt), L2, nst);
        const float pp = ex2(e.x);
        return __fmul_rn(pp, fmaf(h, sgn_pq(pp, ex2(e.y)), c0));
      };
      auto step3 = [&](auto&& cs, auto&& ct, auto n, int q) {
        TG* gq = gmine + int64_t(q) * kStepVecs * VE;
        if (bad) {  // out-of-range target: the whole gradient row is NaN
          float nan[VE];
#pragma unroll
          for (int j = 0; j < VE; ++j) nan[j] = __uint_as_float(0x7fc00000u);
#pragma unroll
          for (int u = 0; u < kPS; ++u)
            if (u < int(n)) store_grad<T, TG, VE>(gq + u * NT * VE, nan, drop);
          return;
        }
        if (from_bits) {
          // this step's bits at the top of the word's slot for it
          const uint32_t word = sbits[(q / kSpw) * NT + tid] << ((q % kSpw) * kBits);
#pragma unroll
          for (int u = 0; u < kPS; ++u) {
            if (u < int(n)) {
              float xs[VE], g[VE];
              unpack_raw<T, VE>(cs(u), xs);
#pragma unroll
              for (int j = 0; j < VE; j += 2) {
                const float2 e = __ffma2_rn(make_float2(xs[j], xs[j + 1]), L2, ns22);
                const int b0 = 31 - (u * VE + j);
                const float ca = ((word >> b0) & 1u) ? c_minus : c_plus;
                const float cb = ((word >> (b0 - 1)) & 1u) ? c_minus : c_plus;
                const float2 gg =
                    __fmul2_rn(make_float2(ex2(e.x), ex2(e.y)), make_float2(ca, cb));
                g[j] = gg.x;
                g[j + 1] = gg.y;
              }
              store_grad<T, TG, VE>(gq + u * NT * VE, g, drop);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < kPS; ++u) {
            if (u < int(n)) {
              // the teacher comes from the ring unless step 3 was planned on
              // sign bits (then it was not staged: read it from L2 / HBM)
              const uint4 wt = use_bits ? load_raw<T, VE>(tmine + int64_t(q * kPS + u) * NT * VE, drop)
                                        : ct(u);
              float xs[VE], xt[VE], g[VE];
              unpack_raw<T, VE>(cs(u), xs);
              unpack_raw<T, VE>(wt, xt);
#pragma unroll
              for (int j = 0; j < VE; ++j) g[j] = grad_of(xs[j], xt[j]);
              store_grad<T, TG, VE>(gq + u * NT * VE, g, drop);
            }
          }
        }
      };
      pass3(step3);
      if (tail0 + tid < p.V) {
        const int64_t v = tail0 + tid;
        float g = grad_of(Elem<T>::load1(srow + v), Elem<T>::load1(trow + v));
        if (v == tg) g = __fsub_rn(g, gce);
        Elem<TG>::store1(grow + v, bad ? __uint_as_float(0x7fc00000u) : g);
      }
      // the target element, after this thread's vector store of it
      if (owner) Elem<TG>::store1(grow + tg, __fsub_rn(grad_of(xs_tg, xt_tg), gce));
    }
  }
  if (tid == 0 && abort_flag && p.dev_status) atomicOr(p.dev_status, FCT_DEV_WAIT_TIMEOUT);
}

// ===================================================================== scalar path
//
// Rows whose pointers or strides are not 16-byte aligned: plain element
// loads, same arithmetic and reductions.

constexpr int kScalarThreads = 512;

template <typename T, int C, bool kTvd>
__global__ void __launch_bounds__(kScalarThreads, 1) forward_scalar(FwdArgs p) {
  constexpr int NT = kScalarThreads;
  __shared__ float4 red_lse[kMaxWarps];
  __shared__ float2 red_sum[kMaxWarps];
  __shared__ float4 part_lse;
  __shared__ float2 part_sum;

  const int rank = (C > 1) ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
  const int64_t cluster_id = blockIdx.x / C;
  const int64_t n_clusters = gridDim.x / C;
  const int64_t per = (p.V + C - 1) / C;
  const int64_t vb = min(p.V, rank * per);
  const int64_t ve = min(p.V, vb + per);
  const T* S = static_cast<const T*>(p.student);
  const T* Tt = static_cast<const T*>(p.teacher);

  for (int64_t row = cluster_id; row < p.BT; row += n_clusters) {
    const int64_t tg = p.target[row];
    if (tg == p.ignore_index) {
      if (rank == 0 && threadIdx.x == 0) write_ignored<kTvd>(p, row);
      continue;
    }
    const T* srow = S + row * p.ld_s;
    const T* trow = kTvd ? Tt + row * p.ld_t : nullptr;
    Lse2 a = lse2_empty(), b = lse2_empty();
    for (int64_t v = vb + threadIdx.x; v < ve; v += NT) {
      float xs[1] = {Elem<T>::load1(srow + v)};
      lse2_update(a, xs);
      if constexpr (kTvd) {
        float xt[1] = {Elem<T>::load1(trow + v)};
        lse2_update(b, xt);
      }
    }
    block_merge2<NT>(a, b, red_lse);
    cluster_merge2<C>(a, b, &part_lse);
    const float lse_s = lse2_finish(a);
    if constexpr (!kTvd) {
      if (rank == 0 && threadIdx.x == 0) {
        const float s_tg = (tg >= 0 && tg < p.V) ? Elem<T>::load1(srow + tg) : 0.f;
        write_row<false>(p, row, tg, lse_s, 0.f, 0.f, 0.f, s_tg);
      }
      if constexpr (C > 1) {
        cluster_sync_all();
      } else {
        __syncthreads();
      }
    } else {
      const float lse_t = lse2_finish(b);
      const float ns2 = -(lse_s * kLog2e);
      const float nt2 = -(lse_t * kLog2e);
      float sig_p = 0.f, sig_q = 0.f;
      for (int64_t v = vb + threadIdx.x; v < ve; v += NT)
        tvd_accum1(Elem<T>::load1(srow + v), Elem<T>::load1(trow + v), ns2, nt2, sig_p, sig_q);
      float abs_sum = sig_p - sig_q;  // sum |p - q| = sum (p - q) * sign(p - q)
      float sig = sig_p;
      block_sum2<NT>(abs_sum, sig, red_sum);
      cluster_sum2<C>(abs_sum, sig, &part_sum, rank);
      if (rank == 0 && threadIdx.x == 0) {
        const float s_tg = (tg >= 0 && tg < p.V) ? Elem<T>::load1(srow + tg) : 0.f;
        write_row<true>(p, row, tg, lse_s, lse_t, abs_sum, sig, s_tg);
      }
    }
  }
  if constexpr (C > 1) cluster_sync_all();
}

// ===================================================================== launch

template <typename K>
cudaError_t launch_cluster(K kernel, int C, int nt, size_t smem, int n_clusters,
                           const FwdArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_clusters * C));
  cfg.blockDim = dim3(nt);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <typename K>
int max_clusters(K kernel, int C, int nt, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C * 64);
  cfg.blockDim = dim3(nt);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  return n > 0 ? n : 1;
}

// One-time set-up of a kernel configuration on each device: the shared-memory
// opt-in is a per-device property of the function, and the occupancy query
// is answered for the current device.
struct PerDevice {
  std::mutex mu;
  int value[64];
  bool done[64] = {};
};

template <class Init>
int per_device(PerDevice& c, Init&& init) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lk(c.mu);
  if (!c.done[dev]) {
    c.value[dev] = init();
    c.done[dev] = true;
  }
  return c.value[dev];
}

// Start stagger of the multi-pass kernels: the clusters' start times are
// spread, in kStaggerGroups interleaved groups, over plan.stagger times an
// estimate of one row's time (about 0.1 clock cycles per byte a CTA reads in
// one pass of a row, measured on GB300 for the single launch at V = 151936
// bf16), when every cluster has at least kStaggerMinRows rows (with one row
// each, the last group's wait costs more than the spread saves).  Measured
// at 8192 x 151936 bf16, against starting together: a spread of half a
// row's time in 8 interleaved groups, one launch 1.619 -> 1.582 ms and the
// forward alone 2.130 -> 2.084 ms with its backward; a whole row's time,
// 1.579 and 2.100; the same spreads over contiguous ranges of clusters
// gained about half as much.  With few rows per CTA (bulk-copy ring, V =
// 151936 bf16, single launch): 304 rows 0.0865 -> 0.0785 ms, 608 rows
// 0.159 -> 0.145, 1216 rows 0.281 -> 0.251, 2048 rows 0.443 -> 0.408; one
// row per CTA (152 rows) 0.0527 -> 0.0564, hence at least 2.
// Cross-entropy alone on clusters (fp32 rows of V = 256000 on 2-CTA
// clusters) measured slower staggered at few rows per cluster (304 rows
// 0.115 -> 0.121 ms, 1024 rows 0.373 -> 0.389), so it keeps the earlier
// threshold of 32.
constexpr double kStaggerCyclesPerByte = 0.1;
constexpr int kStaggerMinRows = 2, kStaggerMinRowsCeCluster = 32;

// One (kernel, configuration) instance: shared-memory opt-in and the
// occupancy query are done once per device.
template <typename T, int VE, int C, bool kTvd, bool kGrad, int NT, typename TG, bool kSigns>
cudaError_t run_pipelined(const FwdArgs& a, int n_slots, double stagger, cudaStream_t st) {
  constexpr size_t kSmem = size_t(kStages) * (kTvd ? 2 : 1) * kPerStep * NT * 16 +
                           ((kGrad && kTvd) ? size_t(kMaxSignWords) * NT * 4 : 0);
  auto kernel = forward_pipelined<T, VE, C, kTvd, kGrad, NT, TG, kSigns>;
  static PerDevice cache;
  const int n_max = per_device(cache, [&] {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmem)) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    return max_clusters(kernel, C, NT, kSmem);
  });
  if (n_max < 0) return cudaErrorInvalidConfiguration;
  int n = n_max;
  if (n_slots > 0 && n > n_slots) n = n_slots;
  if (n > a.BT) n = static_cast<int>(a.BT);
  FwdArgs b = a;
  if constexpr (kTvd || kGrad) {  // several passes per row: stagger the clusters' start
    constexpr int kMinRows = (!kTvd && C > 1) ? kStaggerMinRowsCeCluster : kStaggerMinRows;
    if (a.BT >= int64_t(kMinRows) * n) {
      const double row_bytes = (kTvd ? 2.0 : 1.0) * double(a.V) * double(sizeof(T)) / C;
      b.stagger = static_cast<int64_t>(stagger * kStaggerCyclesPerByte * row_bytes);
    }
  }
  return launch_cluster(kernel, C, NT, kSmem, n, b, st);
}

// The bulk-copy ring form: one CTA per row, 512 consumers plus a producer
// warp; steps of 4 vectors per thread and tensor (32 KB per tensor), 3 slots,
// each released after the warps have computed on it; the forward alone asks
// L2 for its first pass 4 steps ahead of the ring (measured at 8192 x 151936
// bf16: forward 0.956 -> 0.942 ms; the single launch was 1% slower with it).
// Smaller steps with more slots, releasing slots before computing, and 480
// consumers were all measured slower or equal.
// Steps carried between passes (RingPlan): step 2's last 3 steps into step 3
// (measured at 8192 x 151936 bf16: single launch 1.487 -> 1.474 ms, results
// unchanged); none from step 1 into step 2 (carrying 1 or 2 steps made the
// forward alone 0.4-0.8% faster but the single launch 1% slower, and both
// must share step 2's order to agree bit for bit).
constexpr int kTmaThreads = 512, kTmaPerStep = 4, kTmaStages = 3;
constexpr int kTmaCarry1 = 0, kTmaCarry3 = 3;

template <typename T, bool kGrad, typename TG = T, bool kSigns = false, bool kLseIn = false>
cudaError_t run_tma(const FwdArgs& a, const FwdPlan& plan, cudaStream_t st) {
  constexpr int NT = kTmaThreads;
  constexpr int VE = Elem<T>::kVec;
  constexpr size_t kSmem = size_t(kTmaStages) * 2 * kTmaPerStep * NT * 16 +
                           (kGrad ? size_t(kMaxSignWords) * NT * 4 : 0);
  constexpr int kPref = kGrad ? 0 : 4;
  auto kernel = forward_tma<T, VE, kGrad, NT, TG, kTmaPerStep, kTmaStages, kPref, kSigns, kLseIn,
                            kTmaCarry1, kTmaCarry3>;
  static PerDevice cache;
  const int n_max = per_device(cache, [&] {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmem)) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
    return max_clusters(kernel, 1, NT + 32, kSmem);
  });
  if (n_max < 0) return cudaErrorInvalidConfiguration;
  int n = n_max;
  if (plan.slots > 0 && n > plan.slots) n = plan.slots;
  if (n > a.BT) n = static_cast<int>(a.BT);
  FwdArgs b = a;
  if (a.BT >= int64_t(kStaggerMinRows) * n)
    b.stagger = static_cast<int64_t>(plan.stagger * kStaggerCyclesPerByte * 2.0 * double(a.V) *
                                     double(sizeof(T)));
  return launch_cluster(kernel, 1, NT + 32, kSmem, n, b, st);
}

template <typename T, int C, bool kTvd>
cudaError_t run_scalar(const FwdArgs& a, int n_slots, cudaStream_t st) {
  auto kernel = forward_scalar<T, C, kTvd>;
  static PerDevice cache;
  const int n_max = per_device(cache, [&] { return max_clusters(kernel, C, kScalarThreads, 0); });
  if (n_max < 0) return cudaErrorInvalidDevice;
  int n = n_max;
  if (n_slots > 0 && n > n_slots) n = n_slots;
  if (n > a.BT) n = static_cast<int>(a.BT);
  return launch_cluster(kernel, C, kScalarThreads, 0, n, a, st);
}

template <typename T, int C, bool kTvd, bool kGrad, typename TG, bool kSigns>
cudaError_t run(const FwdArgs& a, const FwdPlan& plan, cudaStream_t st) {
  constexpr int VE = Elem<T>::kVec;
  if constexpr (kGrad) {
    if (!plan.vec) return cudaErrorInvalidValue;  // the host routes this case to two launches
  } else {
    if (!plan.vec) return run_scalar<T, C, kTvd>(a, plan.slots, st);
  }
  return run_pipelined<T, VE, C, kTvd, kGrad, 512, TG, kSigns>(a, plan.slots, plan.stagger, st);
}

template <typename T, bool kTvd, bool kGrad, typename TG = T, bool kSigns = false>
cudaError_t run_c(const FwdArgs& a, const FwdPlan& plan, cudaStream_t st) {
  switch (plan.cluster) {
    case 1: return run<T, 1, kTvd, kGrad, TG, kSigns>(a, plan, st);
    case 2: return run<T, 2, kTvd, kGrad, TG, kSigns>(a, plan, st);
    case 4: return run<T, 4, kTvd, kGrad, TG, kSigns>(a, plan, st);
    default: return run<T, 8, kTvd, kGrad, TG, kSigns>(a, plan, st);
  }
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, const FwdPlan& plan, cudaStream_t st) {
  if (a.lse_part_s != nullptr) {
    // step 1 given: the two-pass single launch (one CTA per row: L2 holds
    // only the student between its passes)
    if (!a.grad || !a.tvd || !plan.vec || a.signs || a.lse_part_t == nullptr || a.lse_n <= 0)
      return cudaErrorInvalidValue;
    if (a.dtype == FCT_BF16) return run_tma<bf16_t, true, bf16_t, false, true>(a, plan, st);
    return a.grad_bf16 ? run_tma<float, true, bf16_t, false, true>(a, plan, st)
                       : run_tma<float, true, float, false, true>(a, plan, st);
  }
  if (plan.ring != 1 && plan.vec && plan.cluster == 1 && a.tvd) {
    // the fused forward (alone, with sign words, or with its backward) on the
    // bulk-copy ring: the automatic choice where a row belongs to one CTA
    if (a.signs) {
      if (a.grad) return cudaErrorInvalidValue;
      return a.dtype == FCT_BF16 ? run_tma<bf16_t, false, bf16_t, true>(a, plan, st)
                                 : run_tma<float, false, float, true>(a, plan, st);
    }
    if (a.dtype == FCT_BF16)
      return a.grad ? run_tma<bf16_t, true>(a, plan, st) : run_tma<bf16_t, false>(a, plan, st);
    if (a.grad)
      return a.grad_bf16 ? run_tma<float, true, bf16_t>(a, plan, st)
                         : run_tma<float, true>(a, plan, st);
    return run_tma<float, false>(a, plan, st);
  }
  if (a.signs) {  // the forward alone with sign words (vector path only)
    if (!plan.vec || !a.tvd || a.grad) return cudaErrorInvalidValue;
    return a.dtype == FCT_BF16 ? run_c<bf16_t, true, false, bf16_t, true>(a, plan, st)
                               : run_c<float, true, false, float, true>(a, plan, st);
  }
  if (a.grad && !a.tvd) {  // cross-entropy alone in one launch
    return a.dtype == FCT_BF16 ? run_c<bf16_t, false, true>(a, plan, st)
                               : run_c<float, false, true>(a, plan, st);
  }
  if (a.dtype == FCT_BF16) {
    if (a.grad) return run_c<bf16_t, true, true>(a, plan, st);
    return a.tvd ? run_c<bf16_t, true, false>(a, plan, st) : run_c<bf16_t, false, false>(a, plan, st);
  }
  if (a.grad) {
    return a.grad_bf16 ? run_c<float, true, true, bf16_t>(a, plan, st)
                       : run_c<float, true, true>(a, plan, st);
  }
  return a.tvd ? run_c<float, true, false>(a, plan, st) : run_c<float, false, false>(a, plan, st);
}

}  // namespace fct
