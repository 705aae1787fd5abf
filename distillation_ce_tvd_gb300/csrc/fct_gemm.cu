// bf16 GEMM on the fifth-generation tensor cores: C (+)= A * B^T.
//
// The fused-linear loss computes logits from hidden states and lm_head
// weights and, backwards, the gradients of both: dense contractions (the
// Liger-Kernel overview's fused linear cross-entropy computes logits block by
// block and never holds the whole (BT, V) logit matrix).  This kernel is
// their GB300 form:
//   * operands: A is M x K and B is N x K (C(m, n) = sum_k A(m, k) B(n, k)),
//     bf16, each either K-major (A(m, k) at a[m * ld + k]) or MN-major
//     (A(m, k) at a[k * ld + m]), so the products with a transposed operand
//     (d hidden = G W, d weight = G^T H) need no transposed copies;
//   * a cluster of two CTAs on an SM pair computes one 256 x 256 tile of C
//     with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16 per
//     instruction, bf16 x bf16, fp32 accumulate): each CTA stages, by TMA
//     (cp.async.bulk.tensor, 128-byte swizzle), its own 128 rows of A and its
//     half (128 rows) of B, 64 K-columns per stage, 6 stages deep, and holds
//     the accumulator of its 128 rows in its own tensor memory.  Against one
//     CTA computing 128 x 256 alone, each SM stages 32 KB per K block
//     instead of 48 KB for the same tensor-core work;
//   * two accumulators of 256 columns per CTA (512 columns), so the epilogue
//     of one tile overlaps the MMAs of the next; four warps per CTA read
//     theirs with tcgen05.ld (each its 32-lane quarter, one output row per
//     thread) and store fp32 or bf16 rows, or add into an fp32 C;
//   * a persistent grid of as many pairs as fit, walking the tiles along the
//     index of the smaller operand first (M tiles of one N column when A is
//     the smaller one), so pairs working at once share the larger operand's
//     tile through L2 and the smaller operand stays there whole.
// Per CTA: warp 0 issues TMA, warp 1 owns the tensor memory (and, in the
// pair's rank-0 CTA, issues the MMAs), warps 2-5 run the epilogue.  Every
// mbarrier wait is bounded: a wait that runs out sets an abort flag, the
// roles stop, the last copies and MMAs are waited for (bounded) before the
// tensor memory is freed, and the kernel ORs FCT_DEV_WAIT_TIMEOUT into the
// status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

namespace {

constexpr int kCtaRows = 128;  // rows of A and of B each CTA of a pair stages
constexpr int kBM = 256, kBN = 256, kBK = 64;  // the pair's tile
constexpr int kGStages = 6;
constexpr int kGemmThreads = 192;
constexpr uint32_t kHalfBytes = kCtaRows * kBK * 2;  // 16 KB: one operand's rows of a CTA
constexpr uint32_t kGStageBytes = 2 * kHalfBytes;     // A and B rows of a CTA
constexpr uint32_t kBoxBytes = 64 * kBK * 2;          // one 64 x 64 box of an MN-major operand
constexpr uint32_t kTmemCols = 2 * kBN;               // two fp32 accumulators of 256 columns
// Epilogue staging: per epilogue warp two buffers of 32 rows x 128 bytes
// (32 fp32 or 64 bf16 columns), written in the 128-byte swizzle of the C
// tensor map and sent out by TMA.
constexpr uint32_t kOutBufBytes = 32 * 128;
constexpr uint32_t kEpiBytes = 4 * 2 * kOutBufBytes;  // 32 KB
constexpr size_t kGemmSmem =
    size_t(kGStages) * kGStageBytes + kEpiBytes + 1024;  // + room to align to 1 KB

// Output kinds: fp32 C, bf16 C, fp32 C accumulated into, and fp32 or bf16
// C with each row's base-2 log-sum-exp state over each 256-column tile
// (GemmArgs::lse_part), taken on the values as stored.
static_assert(kBN == kGemmLseTile, "one log-sum-exp state per pair tile column block");

enum COut { kOutF32 = 0, kOutBf16 = 1, kOutAddF32 = 2, kOutF32Lse = 3, kOutBf16Lse = 4 };
template <int kOut>
constexpr bool kBf16C = kOut == kOutBf16 || kOut == kOutBf16Lse;
template <int kOut>
constexpr bool kLseC = kOut == kOutF32Lse || kOut == kOutBf16Lse;

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B bf16 (bits 7-9 and 10-12 = 1), A and B major-ness
// (bits 15 and 16: 0 K-major, 1 MN-major), N / 8 at bits 17-22, M / 16 at
// bits 24-28.
template <bool kAmn, bool kBmn>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kAmn) << 15) | (uint32_t(kBmn) << 16) |
         (uint32_t(kBN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
}

// Shared-memory matrix descriptor of a tile written by TMA with 128-byte
// swizzle (8-row atoms of 128-byte rows, 1024 bytes): start address, leading
// and stride byte offsets in 16-byte units, version 1 (bits 46-47), swizzle
// mode 2 = 128-byte (bits 61-63).
//   K-major: rows are the M (N) index, 64 K elements per row; atoms of 8
//   rows are 1024 bytes apart (stride offset); the leading offset is unused.
//   A K step of 16 advances the start by 32 bytes inside the atom.
//   MN-major: rows are the K index, 64 M (N) elements per row; atoms of 8 K
//   rows are 1024 bytes apart (stride offset), the next 64 M (N) elements
//   start one 64 x 64 box later (leading offset 8192 bytes).  A K step of 16
//   advances the start by 16 rows = 2048 bytes.
template <bool kMn>
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(kMn ? (kBoxBytes >> 4) : 1u) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}
template <bool kMn>
__host__ __device__ constexpr uint64_t desc_k_step() {  // one K step of 16 elements, in 16-byte units
  return kMn ? (16 * 128) >> 4 : (16 * 2) >> 4;
}

// A 2-D TMA load into this CTA's shared memory whose completion is counted
// on the mbarrier at cluster address `bar` (the pair's rank-0 CTA's).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// A CTA's rows of an operand for k block kb: rows r0 .. r0 + 127 of the M (N)
// index.  K-major: one box {64 K, 128}.  MN-major: two boxes {64 M (N),
// 64 K}, 8 KB apart.
template <bool kMn>
__device__ __forceinline__ void load_rows(uint32_t dst, const CUtensorMap* map, int r0, int kb,
                                          uint32_t bar) {
  if constexpr (kMn) {
#pragma unroll
    for (int j = 0; j < kCtaRows / 64; ++j)
      tma_load_2d(dst + j * kBoxBytes, map, r0 + 64 * j, kb * kBK, bar);
  } else {
    tma_load_2d(dst, map, kb * kBK, r0, bar);
  }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The cluster address of this CTA's shared variable at `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <uint32_t kIdesc>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier at `bar`'s offset in both CTAs of the pair
// when every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns of tensor memory: thread i of the
// warp receives lane (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct GemmArgs {
  int64_t M, N, K;
  void* C;
  int64_t ldc;
  int vec;    // C's rows start on 16-byte boundaries: vector stores
  int tma_c;  // C written through its tensor map (TMA store / reduce-add)
  int n_fast; // tile walk: N index fastest (A is the larger operand) or M fastest
  // split K: unit u covers tile u % tiles and the K blocks of part
  // u / tiles; part s writes its fp32 partial tile to rows
  // s * slab_rows + m of C (slab_rows >= the M tiles' extent)
  int splits;
  int k_per;  // K blocks per part
  int64_t slab_rows;
  int32_t* status;
  // lse kinds: row r's state over tile column block t at lse_part[r * lse_ld + t]
  float2* lse_part;
  int64_t lse_ld;
};

// Folds n values (n <= kN; the first n are columns inside C) into a running
// base-2 log-sum-exp state (m2, s): the same representation and rounding
// steps as the loss kernel's step 1 (m2 = max x * log2 e, s = sum of
// 2^(x log2 e - m2)), one rescale per call.  Full groups (n == kN, all but
// a row's last tile) take three-input maxima and packed f32x2 FMAs and adds.
template <int kN>
__device__ __forceinline__ void lse_fold(float& m2, float& s, const float (&x)[kN], int n) {
  static_assert(kN % 4 == 0, "groups of four");
  float vm = -INFINITY;
  if (n >= kN) {
#pragma unroll
    for (int j = 0; j < kN; j += 2) vm = max3(vm, x[j], x[j + 1]);
  } else {
#pragma unroll
    for (int j = 0; j < kN; ++j)
      if (j < n) vm = fmaxf(vm, x[j]);
  }
  const float m2n = vm * kLog2e;
  if (m2n > m2) {
    s *= ex2(m2 - m2n);
    m2 = m2n;
  }
  const float2 L2 = make_float2(kLog2e, kLog2e), nm = make_float2(-m2, -m2);
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  if (n >= kN) {
#pragma unroll
    for (int j = 0; j < kN; j += 4) {
      const float2 e0 = __ffma2_rn(make_float2(x[j], x[j + 1]), L2, nm);
      const float2 e1 = __ffma2_rn(make_float2(x[j + 2], x[j + 3]), L2, nm);
      a0 = __fadd2_rn(a0, make_float2(ex2(e0.x), ex2(e0.y)));
      a1 = __fadd2_rn(a1, make_float2(ex2(e1.x), ex2(e1.y)));
    }
  } else {
#pragma unroll
    for (int j = 0; j < kN; ++j)
      if (j < n) a0.x += ex2(fmaf(x[j], kLog2e, -m2));
  }
  s += (a0.x + a0.y) + (a1.x + a1.y);
}

// Tile t's (M tile, N tile).  Pairs working at once take consecutive t, so
// they share the operand tile of the slow index through L2; the fast index
// runs over the smaller operand, which stays in L2 as a whole.
__device__ __forceinline__ void tile_mn(const GemmArgs& g, int64_t t, int64_t m_tiles,
                                        int64_t n_tiles, int64_t& tm, int64_t& tn) {
  if (g.n_fast) {
    tn = t % n_tiles;
    tm = t / n_tiles;
  } else {
    tm = t % m_tiles;
    tn = t / m_tiles;
  }
}

// TMA from this CTA's shared memory to C: a plain store, or an fp32 add
// performed at L2 (the read-modify-write of an accumulated C never reaches
// the SM).  Completion is tracked per thread in bulk groups.
template <bool kAdd>
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  if constexpr (kAdd)
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%1, %2}], [%3];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most one (none) of this thread's bulk groups still reads
// shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// One thread's 128-byte row of a staging buffer, 16-byte chunk j at chunk
// position j ^ (row % 8): the 128-byte swizzle of the C tensor map, which
// also spreads a warp's chunk stores over all banks.
__device__ __forceinline__ void stage_row(uint32_t buf, int row, const uint32_t (&w)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = buf + uint32_t(row) * 128u + uint32_t((j ^ (row & 7)) * 16);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[4 * j]),
                 "r"(w[4 * j + 1]), "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                 : "memory");
  }
}

// Stores (or adds) 32 consecutive fp32 results of one C row, columns
// [col0, col0 + 32) clipped to N.
template <int kOut>
__device__ __forceinline__ void store_row32(const GemmArgs& g, int64_t row, int64_t col0,
                                            const uint32_t (&r)[32]) {
  if constexpr (kBf16C<kOut>) {
    uint16_t* crow = static_cast<uint16_t*>(g.C) + row * g.ldc + col0;
    if (g.vec && col0 + 32 <= g.N) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        const uint4 v = make_uint4(pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                                   pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                                   pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5])),
                                   pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7])));
        *reinterpret_cast<uint4*>(crow + j) = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < g.N)
          crow[j] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(r[j]), 0.f) & 0xffffu);
    }
  } else {
    float* crow = static_cast<float*>(g.C) + row * g.ldc + col0;
    if (g.vec && col0 + 32 <= g.N) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                               __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        if constexpr (kOut == kOutAddF32) {
          const float4 o = *reinterpret_cast<const float4*>(crow + j);
          v.x = o.x + v.x;
          v.y = o.y + v.y;
          v.z = o.z + v.z;
          v.w = o.w + v.w;
        }
        *reinterpret_cast<float4*>(crow + j) = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col0 + j >= g.N) continue;
        const float v = __uint_as_float(r[j]);
        crow[j] = (kOut == kOutAddF32) ? crow[j] + v : v;
      }
    }
  }
}

template <bool kAmn, bool kBmn, int kOut>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, GemmArgs g) {
  extern __shared__ uint8_t gemm_smem[];
  // full_bar: used in the rank-0 CTA only (both CTAs' copies count on it);
  // acc_empty: rank 0's counts the epilogue warps of both CTAs
  __shared__ __align__(8) uint64_t full_bar[kGStages], empty_bar[kGStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const uint32_t smem0 = (smem_addr(gemm_smem) + 1023u) & ~1023u;
  const int64_t m_tiles = (g.M + kBM - 1) / kBM, n_tiles = (g.N + kBN - 1) / kBN;
  const int64_t tiles = m_tiles * n_tiles;
  const int64_t units = tiles * g.splits;
  const int k_iters = static_cast<int>((g.K + kBK - 1) / kBK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);
    }
    mbar_init(&done_bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's tensor memory
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any copy or arrive
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t full0 = map_to_rank(smem_addr(&full_bar[0]), 0);
  const uint32_t acc_empty0 = map_to_rank(smem_addr(&acc_empty[0]), 0);

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int64_t u = pair; ok && u < units; u += n_pairs) {
        int64_t tm, tn;
        tile_mn(g, u % tiles, m_tiles, n_tiles, tm, tn);
        const int m0 = static_cast<int>(tm * kBM) + int(rank) * kCtaRows;
        const int n0 = static_cast<int>(tn * kBN) + int(rank) * kCtaRows;
        const int kb0 = static_cast<int>(u / tiles) * g.k_per;
        const int kb1 = min(k_iters, kb0 + g.k_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * kGStageBytes);
          const uint32_t sa = smem0 + stage * kGStageBytes;
          load_rows<kAmn>(sa, &tmA, m0, kb, full0 + 8u * stage);
          load_rows<kBmn>(sa + kHalfBytes, &tmB, n0, kb, full0 + 8u * stage);
          ++issued;
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the last fills of both CTAs have landed before the leader's producer
      // leaves (its full barriers count the peer's bytes too; bounded, even
      // after an abort)
      if (leader)
        for (uint32_t i = (issued > uint32_t(kGStages) ? issued - kGStages : 0); i < issued; ++i)
          mbar_wait(&full_bar[i % kGStages], (i / kGStages) & 1u, &abort_flag, false);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {  // ---- MMA issuer for the pair
      constexpr uint32_t kId = idesc<kAmn, kBmn>();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int64_t local = 0;
      for (int64_t u = pair; ok && u < units; u += n_pairs, ++local) {
        const int acc = static_cast<int>(local & 1);
        const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, &abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + uint32_t(acc * kBN);
        const int kb0 = static_cast<int>(u / tiles) * g.k_per;
        const int kb1 = min(k_iters, kb0 + g.k_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem0 + stage * kGStageBytes;
          const uint64_t adesc = smem_desc<kAmn>(sa), bdesc = smem_desc<kBmn>(sa + kHalfBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16<kId>(d, adesc + kk * desc_k_step<kAmn>(), bdesc + kk * desc_k_step<kBmn>(),
                           (kb > kb0 || kk > 0) ? 1u : 0u);
          umma_commit_pair(&empty_bar[stage]);  // both CTAs' stages are free once these are done
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(&acc_full[acc]);
      }
      umma_commit_pair(&done_bar);  // every MMA issued has completed
    }
  } else {  // ---- epilogue: warps 2-5 of each CTA, each its 32-lane quarter
    const int q = warp & 3;
    int64_t local = 0;
    bool last_sent = false;  // lane 0: whether the previous block committed a bulk group
    for (int64_t u = pair; u < units; u += n_pairs, ++local) {
      const int acc = static_cast<int>(local & 1);
      const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
      // the warp agrees on the outcome, so the .sync.aligned loads below run
      // converged even if a wait ran out on some lanes only
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], acc_phase, &abort_flag))) break;
      tc_fence_after();
      int64_t tm, tn;
      tile_mn(g, u % tiles, m_tiles, n_tiles, tm, tn);
      const int64_t m0 = tm * kBM + int64_t(rank) * kCtaRows;
      const int64_t n0 = tn * kBN;
      const int64_t slab = (u / tiles) * g.slab_rows;  // 0 without split K
      const uint32_t tq = tmem + (uint32_t(q * 32) << 16) + uint32_t(acc * kBN);
      // lse kinds: this thread's row over the tile's columns
      [[maybe_unused]] float lse_m2 = -INFINITY, lse_s = 0.f;
      if (g.tma_c) {
        // 32-row blocks of 128 bytes per row through two staging buffers
        const uint32_t buf0 = smem0 + kGStages * kGStageBytes + uint32_t(q) * 2 * kOutBufBytes;
        constexpr int kCols = kBf16C<kOut> ? 64 : 32;
        const int y = static_cast<int>(slab + m0 + q * 32);
        const int64_t rows_end = slab + (g.splits > 1 ? g.slab_rows : g.M);
#pragma unroll 1
        for (int c = 0; c < kBN / kCols; ++c) {
          uint32_t w[32];
          if constexpr (kBf16C<kOut>) {
            uint32_t r[32];
            tmem_ld32(tq + uint32_t(c * 64), r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              w[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            tmem_ld32(tq + uint32_t(c * 64 + 32), r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              w[16 + j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
          } else {
            tmem_ld32(tq + uint32_t(c * 32), w);
          }
          if constexpr (kLseC<kOut>) {
            const int64_t nv = g.N - (n0 + c * kCols);
            float x[kCols];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if constexpr (kBf16C<kOut>) {
                x[2 * j] = __uint_as_float(w[j] << 16);
                x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
              } else {
                x[j] = __uint_as_float(w[j]);
              }
            }
            lse_fold<kCols>(lse_m2, lse_s, x, nv < kCols ? static_cast<int>(nv) : kCols);
          }
          if (c == kBN / kCols - 1) {  // the accumulator is read: release it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * acc);
          }
          // buffers alternate (kBN / kCols is even, so also across tiles);
          // the store that last used this one has finished reading it
          const uint32_t buf = buf0 + uint32_t(c & 1) * kOutBufBytes;
          if (lane == 0) {
            if (last_sent)
              bulk_wait_read_1();
            else
              bulk_wait_read_0();
          }
          __syncwarp();
          stage_row(buf, lane, w);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            last_sent = n0 + c * kCols < g.N && y < rows_end;
            if (last_sent)
              tma_store_2d<kOut == kOutAddF32>(&tmC, static_cast<int>(n0) + c * kCols, y, buf);
          }
        }
      } else {
        const int64_t row = m0 + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tq + uint32_t(c * 32), r);
          const int64_t col0 = n0 + c * 32;
          if (row < g.M && col0 < g.N) store_row32<kOut>(g, slab + row, col0, r);
          if constexpr (kLseC<kOut>) {
            const int64_t nv = g.N - col0;
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              if constexpr (kBf16C<kOut>) {  // the values as stored
                const uint32_t b = pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                x[j] = __uint_as_float(b << 16);
                x[j + 1] = __uint_as_float(b & 0xffff0000u);
              } else {
                x[j] = __uint_as_float(r[j]);
                x[j + 1] = __uint_as_float(r[j + 1]);
              }
            }
            lse_fold<32>(lse_m2, lse_s, x, nv < 32 ? static_cast<int>(nv) : 32);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * acc);
      }
      if constexpr (kLseC<kOut>) {
        const int64_t row = m0 + q * 32 + lane;
        if (row < g.M) g.lse_part[row * g.lse_ld + tn] = make_float2(lse_m2, lse_s);
      }
    }
    if (lane == 0) bulk_wait_all();  // C is written before the kernel ends
  }
  tc_fence_before();
  __syncthreads();
  // the pair's MMAs have all completed before either CTA frees its tensor
  // memory or leaves (the peer's MMAs read this CTA's shared memory)
  if (warp == 1 && lane == 0) mbar_wait(&done_bar, 0, &abort_flag, false);
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  if (threadIdx.x == 0 && abort_flag && g.status) atomicOr(g.status, FCT_DEV_WAIT_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map of a bf16 operand: `inner` contiguous elements per line, `outer`
// lines ld elements apart; boxes of 64 x box_outer, 128-byte swizzle, zero
// fill outside the matrix.
bool make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t ld,
              uint32_t box_outer) {
  auto encode = encode_fn();
  if (encode == nullptr) return false;
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
  const cuuint32_t box[2] = {64u, box_outer};
  const cuuint32_t elem[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// C's map for the epilogue's stores: M rows of N elements, ldc apart, boxes
// of 32 rows x 128 bytes (32 fp32 or 64 bf16), 128-byte swizzle.
bool make_c_map(CUtensorMap* map, void* C, int64_t M, int64_t N, int64_t ldc, bool bf16) {
  auto encode = encode_fn();
  if (encode == nullptr) return false;
  const size_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(M)};
  const cuuint64_t strides[1] = {cuuint64_t(ldc) * es};
  const cuuint32_t box[2] = {cuuint32_t(128 / es), 32u};
  const cuuint32_t elem[2] = {1, 1};
  return encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                C, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The operand's map: K-major rows x K with boxes {64 K, tile rows};
// MN-major K lines of `rows` elements with boxes {64, 64}.
bool operand_map(CUtensorMap* map, const GemmOperand& x, int64_t rows, int64_t K,
                 uint32_t tile_rows) {
  return x.mn_major ? make_map(map, x.ptr, rows, K, x.ld, 64)
                    : make_map(map, x.ptr, K, rows, x.ld, tile_rows);
}

// Fills a launch configuration for a kernel of this file: clusters of two,
// kGemmThreads threads, kGemmSmem bytes of shared memory.
struct PairLaunch {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  PairLaunch() {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kGemmSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

// Sets the shared-memory limit of one instantiation on the current device
// (once) and returns how many of its pairs can be resident at once (0 on
// failure).
template <bool kAmn, bool kBmn, int kOut>
int prepare(int dev) {
  static std::once_flag once[64];
  static int pairs[64];
  std::call_once(once[dev], [&] {
    auto kernel = gemm_kernel<kAmn, kBmn, kOut>;
    pairs[dev] = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmem)) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    PairLaunch l;
    l.cfg.gridDim = dim3(2 * 64);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &l.cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    pairs[dev] = n;
  });
  return pairs[dev];
}

template <bool kAmn, bool kBmn, int kOut>
cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                     const GemmArgs& g, int max_pairs, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int pairs = prepare<kAmn, kBmn, kOut>(dev);
  if (pairs <= 0) return cudaErrorInvalidConfiguration;
  const int64_t units = ((g.M + kBM - 1) / kBM) * ((g.N + kBN - 1) / kBN) * g.splits;
  int64_t n = units < pairs ? units : pairs;
  if (n > max_pairs) n = max_pairs;
  PairLaunch l;
  l.cfg.gridDim = dim3(static_cast<unsigned>(2 * n));
  l.cfg.stream = st;
  return cudaLaunchKernelEx(&l.cfg, gemm_kernel<kAmn, kBmn, kOut>, ma, mb, mc, g);
}

template <int kOut>
cudaError_t dispatch_major(bool a_mn, bool b_mn, const CUtensorMap& ma, const CUtensorMap& mb,
                           const CUtensorMap& mc, const GemmArgs& g, int max_pairs,
                           cudaStream_t st) {
  if (a_mn) return b_mn ? run_gemm<true, true, kOut>(ma, mb, mc, g, max_pairs, st)
                        : run_gemm<true, false, kOut>(ma, mb, mc, g, max_pairs, st);
  return b_mn ? run_gemm<false, true, kOut>(ma, mb, mc, g, max_pairs, st)
              : run_gemm<false, false, kOut>(ma, mb, mc, g, max_pairs, st);
}

// C (M x N, fp32 or bf16) = the sum of `splits` fp32 partial slabs, added in
// slab order (so the result does not depend on which pair computed which
// part).  Slab s holds row m at slabs[(s * slab_rows + m) * slab_ld].
template <bool kBf16>
__global__ void __launch_bounds__(256)
    split_sum_kernel(const float* __restrict__ slabs, int64_t slab_ld, int64_t slab_rows,
                     int splits, void* C, int64_t ldc, int64_t M, int64_t N) {
  const int64_t per_row = (N + 3) / 4;  // groups of four columns
  const int64_t total = M * per_row;
  const int64_t stride_s = slab_rows * slab_ld;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t m = i / per_row, n = (i - m * per_row) * 4;
    const float* p = slabs + m * slab_ld + n;  // slab rows are 16-byte aligned
    float4 acc = *reinterpret_cast<const float4*>(p);
    for (int sp = 1; sp < splits; ++sp) {
      const float4 v = *reinterpret_cast<const float4*>(p + sp * stride_s);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const float r[4] = {acc.x, acc.y, acc.z, acc.w};
    const int cnt = N - n < 4 ? static_cast<int>(N - n) : 4;
    if constexpr (kBf16) {
      uint16_t* c = static_cast<uint16_t*>(C) + m * ldc + n;
      for (int j = 0; j < cnt; ++j)
        c[j] = static_cast<uint16_t>(pack_bf16x2(r[j], 0.f) & 0xffffu);
    } else {
      float* c = static_cast<float*>(C) + m * ldc + n;
      for (int j = 0; j < cnt; ++j) c[j] = r[j];
    }
  }
}

// Bytes of one part's fp32 slab of an M x N result: rows padded to the M
// tiles' extent, row length to a multiple of 4; 0 if that overflows.
constexpr int kMaxSplits = 8;
size_t split_slab_bytes(int64_t M, int64_t N) {
  const uint64_t rows = uint64_t((M + kBM - 1) / kBM) * kBM, cols = uint64_t((N + 3) / 4 * 4);
  if (rows == 0 || cols == 0 || rows > SIZE_MAX / cols / sizeof(float)) return 0;
  return size_t(rows * cols * sizeof(float));
}

// Parts of K for a GEMM of `tiles` pair tiles: split when the tiles alone
// leave pairs idle in the last round (under 90% of the rounds busy), each
// part keeping at least 16 K blocks, the slabs fitting the workspace, and
// only for a gain of at least 4 points of busy rounds.
int plan_splits(int64_t tiles, int k_iters, int pairs, size_t ws_bytes, size_t slab_bytes) {
  if (pairs <= 0 || slab_bytes == 0) return 1;
  auto busy = [&](int S) {
    const double w = double(tiles) * S / pairs;
    return w / std::ceil(w);
  };
  int best = 1;
  double best_busy = busy(1);
  if (best_busy >= 0.9) return 1;
  for (int S = 2; S <= kMaxSplits; ++S) {
    if (k_iters < 16 * S || slab_bytes > ws_bytes / size_t(S)) break;
    const double b = busy(S);
    if (b > best_busy + 0.04) {
      best = S;
      best_busy = b;
    }
  }
  return best;
}

}  // namespace

bool gemm_operand_ok(const void* p, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(p) % 16) == 0 && ld > 0 && ld % 8 == 0;
}

cudaError_t launch_gemm(const GemmOperand& A, const GemmOperand& B, void* C, int64_t ldc,
                        int c_kind, int64_t M, int64_t N, int64_t K, int32_t* status, int sms,
                        cudaStream_t st, void* split_ws, size_t split_ws_bytes, float2* lse_part,
                        int64_t lse_ld) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (M > kGemmMaxDim || N > kGemmMaxDim || K > kGemmMaxDim) return cudaErrorInvalidValue;
  if (!gemm_operand_ok(A.ptr, A.ld) || !gemm_operand_ok(B.ptr, B.ld) || sms <= 0)
    return cudaErrorInvalidValue;
  if (c_kind < kOutF32 || c_kind > kOutBf16Lse) return cudaErrorInvalidValue;
  const bool lse = c_kind == kOutF32Lse || c_kind == kOutBf16Lse;
  if (lse && (lse_part == nullptr || lse_ld < (N + kBN - 1) / kBN || A.mn_major || B.mn_major))
    return cudaErrorInvalidValue;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  CUtensorMap ma, mb;
  if (!operand_map(&ma, A, M, K, kCtaRows) || !operand_map(&mb, B, N, K, kCtaRows))
    return cudaErrorInvalidValue;
  const int max_pairs = sms / 2 > 0 ? sms / 2 : 1;
  const int64_t m_tiles = (M + kBM - 1) / kBM, n_tiles = (N + kBN - 1) / kBN;
  const int k_iters = static_cast<int>((K + kBK - 1) / kBK);

  // split K into parts whose fp32 partial tiles go to slabs in split_ws
  int splits = 1;
  const int64_t slab_rows = m_tiles * kBM, slab_ld = (N + 3) / 4 * 4;
  if (c_kind != kOutAddF32 && !lse && split_ws != nullptr &&
      reinterpret_cast<uintptr_t>(split_ws) % 16 == 0) {
    int pairs = prepare<false, false, kOutF32>(dev);
    if (pairs > max_pairs) pairs = max_pairs;
    splits = plan_splits(m_tiles * n_tiles, k_iters, pairs, split_ws_bytes,
                         split_slab_bytes(M, N));
  }
  if (splits > 1) {
    const int k_per = (k_iters + splits - 1) / splits;
    splits = (k_iters + k_per - 1) / k_per;  // every part gets at least one K block
    CUtensorMap ms;
    // padded slab rows and row ends: a box clipped at N or at the M tiles'
    // extent stays inside its own slab
    if (!make_c_map(&ms, split_ws, splits * slab_rows, N, slab_ld, false))
      return cudaErrorInvalidValue;
    const GemmArgs g{M, N, K, split_ws, slab_ld, 1, 1, M > N ? 1 : 0, splits, k_per, slab_rows,
                     status, nullptr, 0};
    cudaError_t e = dispatch_major<kOutF32>(A.mn_major, B.mn_major, ma, mb, ms, g, max_pairs, st);
    if (e != cudaSuccess) return e;
    const int64_t groups = M * ((N + 3) / 4);
    int64_t blocks = (groups + 255) / 256;
    if (blocks > int64_t(sms) * 8) blocks = int64_t(sms) * 8;
    if (c_kind == kOutBf16)
      split_sum_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
          static_cast<const float*>(split_ws), slab_ld, slab_rows, splits, C, ldc, M, N);
    else
      split_sum_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
          static_cast<const float*>(split_ws), slab_ld, slab_rows, splits, C, ldc, M, N);
    return cudaGetLastError();
  }

  const bool bf16 = c_kind == kOutBf16 || c_kind == kOutBf16Lse;
  const size_t es = bf16 ? 2 : 4;
  const bool aligned16 =
      reinterpret_cast<uintptr_t>(C) % 16 == 0 && (size_t(ldc) * es) % 16 == 0;
  // TMA stores clip a row at 16-byte granularity: a row whose width is not
  // a multiple of 16 bytes would get the next few elements written too
  CUtensorMap mc;
  memset(&mc, 0, sizeof(mc));
  const bool tma_c = aligned16 && (size_t(N) * es) % 16 == 0 &&
                     make_c_map(&mc, C, M, N, ldc, bf16);
  const GemmArgs g{M, N, K, C, ldc, aligned16 ? 1 : 0, tma_c ? 1 : 0, M > N ? 1 : 0, 1, k_iters,
                   0, status, lse_part, lse_ld};
  switch (c_kind) {
    // the logits product only: both operands K-major
    case kOutF32Lse: return run_gemm<false, false, kOutF32Lse>(ma, mb, mc, g, max_pairs, st);
    case kOutBf16Lse: return run_gemm<false, false, kOutBf16Lse>(ma, mb, mc, g, max_pairs, st);
    case kOutF32: return dispatch_major<kOutF32>(A.mn_major, B.mn_major, ma, mb, mc, g, max_pairs, st);
    case kOutBf16:
      return dispatch_major<kOutBf16>(A.mn_major, B.mn_major, ma, mb, mc, g, max_pairs, st);
    default:
      return dispatch_major<kOutAddF32>(A.mn_major, B.mn_major, ma, mb, mc, g, max_pairs, st);
  }
}

size_t gemm_split_workspace_bytes(int64_t M, int64_t N) {
  const size_t slab = split_slab_bytes(M, N);
  return slab <= SIZE_MAX / kMaxSplits ? size_t(kMaxSplits) * slab : 0;
}

}  // namespace fct
