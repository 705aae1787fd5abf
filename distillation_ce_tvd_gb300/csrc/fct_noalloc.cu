// Fused-linear CE + TVD for callers that must not allocate device memory.
//
// The regular fused-linear entry point needs a caller-provided workspace for
// its logit blocks.  Some callers can do neither at call time: a serving or training
// process whose memory is fixed up front (a caching allocator or a KV cache
// that owns all free HBM, so a cudaMalloc outside it fails or fragments it),
// and code on a path that must not synchronise the device, which cudaMalloc
// and cudaFree may do.  This variant computes the same loss and gradients
// with no allocation per call:
//   * its logit blocks live in a fixed array of device memory that is part of
//     this file's module (kScratchBytes below; the driver reserves it on each
//     device when the module loads there and keeps it until the process
//     exits);
//   * its GEMMs run on the library's tensor-core GEMM (which allocates
//     nothing) when the hidden states and weights have 16-byte aligned rows,
//     else on a tiled CUDA-core kernel of its own (fp32 accumulation);
//   * the loss itself is the same single-launch forward + backward kernel
//     as every other path, and the logit gradient is rounded to bf16 the same
//     way before the gradient GEMMs.
// Rows go through in blocks of kScratchBytes / (2 * 4 * round8(V)) rows.
//
// Set-up: the first call on a device looks up the array's device address
// with cudaGetSymbolAddress (with that device current) and queries the
// device; later calls on that device reuse both.  All calls share the array,
// so calls whose work can overlap on the GPU (other streams, other threads)
// race on it; the caller orders them.  Nothing in it has to start at zero:
// each block writes its logits before anything reads them.
#include <mutex>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace {

constexpr size_t kScratchBytes = FCT_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte blocks");

}  // namespace

// Student and teacher fp32 logit blocks; the bf16 logit gradient reuses the
// teacher half.
static __device__ __align__(256) float fct_noalloc_scratch[kScratchBytes / sizeof(float)];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array on `device` (which must be current).
int scratch_on(int device, void** out) {
  if (device < 0 || device >= 64) return FCT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, fct_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FCT_ERR_CUDA;
    }
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return FCT_OK;
}

// ------------------------------------------------------------------ tiled GEMM
//
// C(m, n) = beta * C(m, n) + sum_k A(m, k) * B(k, n) for bf16 A and B given
// by element strides, accumulated in fp32 in increasing k; C fp32, or bf16
// (rounded to nearest even, beta ignored).  64 x 64 output tiles, k in slices
// of 16 staged through shared memory; thread (tx, ty) owns rows ty + 16 i and
// columns tx + 16 j.  Every global access is bounds-checked.
constexpr int kT = 64, kKs = 16, kGemmThreads = 256;

struct Gemm {
  const uint16_t* A;
  int64_t sam, sak;
  const uint16_t* B;
  int64_t sbk, sbn;
  void* C;
  int64_t scm, scn;
  int64_t M, N, K;
  float beta;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

template <bool kBf16Out>
__global__ void __launch_bounds__(kGemmThreads) tiled_gemm(Gemm g) {
  __shared__ float As[kKs][kT + 1];
  __shared__ float Bs[kKs][kT + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t tiles_m = (g.M + kT - 1) / kT, tiles_n = (g.N + kT - 1) / kT;
  for (int64_t tm = blockIdx.y; tm < tiles_m; tm += gridDim.y) {
    for (int64_t tn = blockIdx.x; tn < tiles_n; tn += gridDim.x) {
      const int64_t m0 = tm * kT, n0 = tn * kT;
      float acc[4][4] = {};
      for (int64_t k0 = 0; k0 < g.K; k0 += kKs) {
        // the unit-stride index runs fastest across threads
        for (int i = threadIdx.x; i < kT * kKs; i += kGemmThreads) {
          const int mm = (g.sak == 1) ? i / kKs : i % kT;
          const int kk = (g.sak == 1) ? i % kKs : i / kT;
          const int64_t m = m0 + mm, k = k0 + kk;
          As[kk][mm] = (m < g.M && k < g.K) ? bf16_bits_to_f32(g.A[m * g.sam + k * g.sak]) : 0.f;
        }
        for (int i = threadIdx.x; i < kT * kKs; i += kGemmThreads) {
          const int nn = (g.sbn == 1) ? i % kT : i / kKs;
          const int kk = (g.sbn == 1) ? i / kT : i % kKs;
          const int64_t n = n0 + nn, k = k0 + kk;
          Bs[kk][nn] = (n < g.N && k < g.K) ? bf16_bits_to_f32(g.B[k * g.sbk + n * g.sbn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kKs; ++kk) {
          float a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
          for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
          if (m >= g.M || n >= g.N) continue;
          const int64_t off = m * g.scm + n * g.scn;
          if constexpr (kBf16Out) {
            static_cast<uint16_t*>(g.C)[off] =
                static_cast<uint16_t>(fct::pack_bf16x2(acc[i][j], 0.f) & 0xffffu);
          } else {
            float* c = static_cast<float*>(g.C) + off;
            *c = (g.beta == 0.f) ? acc[i][j] : fmaf(g.beta, *c, acc[i][j]);
          }
        }
      }
    }
  }
}

template <bool kBf16Out>
cudaError_t gemm(const Gemm& g, cudaStream_t st) {
  const int64_t tm = (g.M + kT - 1) / kT, tn = (g.N + kT - 1) / kT;
  const dim3 grid(static_cast<unsigned>(tn < 65535 ? tn : 65535),
                  static_cast<unsigned>(tm < 65535 ? tm : 65535));
  tiled_gemm<kBf16Out><<<grid, kGemmThreads, 0, st>>>(g);
  return cudaGetLastError();
}

// fp32 (rows, cols) -> bf16 (rows, cols), both with row stride ld elements,
// rounded to nearest even.
constexpr int kConvThreads = 256;

__global__ void __launch_bounds__(kConvThreads) to_bf16(const float* src, uint16_t* dst,
                                                        int64_t ld, int64_t rows, int64_t cols) {
  const int64_t total = rows * cols;
  for (int64_t i = blockIdx.x * int64_t(kConvThreads) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * kConvThreads) {
    const int64_t r = i / cols, c = i - r * cols;
    dst[r * ld + c] = static_cast<uint16_t>(fct::pack_bf16x2(src[r * ld + c], 0.f) & 0xffffu);
  }
}

// ------------------------------------------------------------------ block loop

// The block loop's GEMMs: the tensor-core GEMM of fct_gemm.cu (no
// allocation either) when every bf16 operand has 16-byte aligned rows, the
// tiled kernel above otherwise.
cudaError_t run_blocks(const fct::LinArgs& a, const fct::FwdPlan& plan, int sms,
                       cudaStream_t st) {
  const bool tc = fct::gemm_operand_ok(a.h_s, a.ld_hs) && fct::gemm_operand_ok(a.w_s, a.ld_ws) &&
                  fct::gemm_operand_ok(a.h_t, a.ld_ht) && fct::gemm_operand_ok(a.w_t, a.ld_wt);
  const int64_t ldl = fct::linear_logits_ld(a.V);
  float* Ls = static_cast<float*>(a.workspace);
  float* Lt = Ls + a.chunk_rows * ldl;
  uint16_t* G = reinterpret_cast<uint16_t*>(Lt);  // bf16 gradient, row stride ldl
  const auto* Hs = static_cast<const uint16_t*>(a.h_s);
  const auto* Ht = static_cast<const uint16_t*>(a.h_t);
  const auto* Ws = static_cast<const uint16_t*>(a.w_s);
  const auto* Wt = static_cast<const uint16_t*>(a.w_t);
  cudaError_t e;
  for (int64_t r0 = 0; r0 < a.BT; r0 += a.chunk_rows) {
    const int64_t R = (a.BT - r0 < a.chunk_rows) ? a.BT - r0 : a.chunk_rows;
    // logits (R x V): A(r, d) = H[r0 + r, d], B(d, v) = W[v, d]
    if (tc) {
      if ((e = fct::launch_gemm(fct::GemmOperand{Hs + r0 * a.ld_hs, a.ld_hs, false},
                                fct::GemmOperand{Ws, a.ld_ws, false}, Ls, ldl, FCT_GEMM_F32, R,
                                a.V, a.d_s, a.dev_status, sms, st)) != cudaSuccess ||
          (e = fct::launch_gemm(fct::GemmOperand{Ht + r0 * a.ld_ht, a.ld_ht, false},
                                fct::GemmOperand{Wt, a.ld_wt, false}, Lt, ldl, FCT_GEMM_F32, R,
                                a.V, a.d_t, a.dev_status, sms, st)) != cudaSuccess)
        return e;
    } else {
      if ((e = gemm<false>(Gemm{Hs + r0 * a.ld_hs, a.ld_hs, 1, Ws, 1, a.ld_ws, Ls, ldl, 1, R,
                                a.V, a.d_s, 0.f},
                           st)) != cudaSuccess)
        return e;
      if ((e = gemm<false>(Gemm{Ht + r0 * a.ld_ht, a.ld_ht, 1, Wt, 1, a.ld_wt, Lt, ldl, 1, R,
                                a.V, a.d_t, 0.f},
                           st)) != cudaSuccess)
        return e;
    }
    // the loss on the block, its logit gradient written over Ls
    fct::FwdArgs f{Ls, Lt, ldl, ldl, FCT_F32, a.target + r0, R, a.V, a.ignore_index,
                   a.ce + r0, a.tvd + r0, a.lse_s + r0, a.lse_t + r0, a.sigma + r0,
                   a.dev_status, Ls, ldl, a.grad_ce + (a.grad_stride ? r0 : 0),
                   a.grad_tvd + (a.grad_stride ? r0 : 0), a.grad_stride,
                   plan.keep_normal ? 1 : 0};
    if ((e = fct::launch_forward(f, plan, st)) != cudaSuccess) return e;
    if (a.grad_h_s == nullptr && a.grad_w_s == nullptr) continue;
    int64_t blocks = (R * a.V + kConvThreads - 1) / kConvThreads;
    if (blocks > int64_t(sms) * 8) blocks = int64_t(sms) * 8;
    to_bf16<<<static_cast<unsigned>(blocks), kConvThreads, 0, st>>>(Ls, G, ldl, R, a.V);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // d hidden (R x D, bf16): A(r, v) = G[r, v], B(v, d) = W[v, d]
    uint16_t* gh = static_cast<uint16_t*>(a.grad_h_s) + r0 * a.ld_ghs;
    if (a.grad_h_s &&
        (e = tc ? fct::launch_gemm(fct::GemmOperand{G, ldl, false},
                                   fct::GemmOperand{Ws, a.ld_ws, true}, gh, a.ld_ghs,
                                   FCT_GEMM_BF16, R, a.d_s, a.V, a.dev_status, sms, st)
                : gemm<true>(Gemm{G, ldl, 1, Ws, a.ld_ws, 1, gh, a.ld_ghs, 1, R, a.d_s, a.V, 0.f},
                             st)) != cudaSuccess)
      return e;
    // d weight (V x D, fp32) += A(v, r) = G[r, v] times B(r, d) = H[r0 + r, d]
    if (a.grad_w_s &&
        (e = tc ? fct::launch_gemm(fct::GemmOperand{G, ldl, true},
                                   fct::GemmOperand{Hs + r0 * a.ld_hs, a.ld_hs, true},
                                   a.grad_w_s, a.ld_gws, FCT_GEMM_ADD_F32, a.V, a.d_s, R,
                                   a.dev_status, sms, st)
                : gemm<false>(Gemm{G, 1, ldl, Hs + r0 * a.ld_hs, a.ld_hs, 1, a.grad_w_s,
                                   a.ld_gws, 1, a.V, a.d_s, R, 1.f},
                              st)) != cudaSuccess)
      return e;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ checks

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
  uintptr_t lo, hi;
};
Span mat_span(const void* p, int64_t rows, int64_t ld, int64_t cols, int64_t e) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * e)};
}
bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

// Whether a (rows, cols) matrix of e-byte elements with row stride ld spans
// at most 2^62 bytes, checked without overflowing, so that every byte range
// computed from the sizes is exact.
bool span_fits(int64_t rows, int64_t ld, int64_t cols, int64_t e) {
  const int64_t lim = (int64_t(1) << 62) / e;
  if (rows <= 0 || cols <= 0 || ld < cols || cols > lim) return false;
  return rows - 1 <= (lim - cols) / ld;
}

int check(const fct::LinArgs& a) {
  if (a.V <= 0 || a.d_s <= 0 || a.d_t <= 0) return FCT_ERR_INVALID_ARG;
  // One student + one teacher fp32 row must fit in the scratch array; test
  // V before any size arithmetic.
  if (a.V > int64_t(kScratchBytes / (2 * sizeof(float)))) return FCT_ERR_UNSUPPORTED;
  if (a.ld_hs < a.d_s || a.ld_ws < a.d_s || a.ld_ht < a.d_t || a.ld_wt < a.d_t)
    return FCT_ERR_INVALID_ARG;
  if ((a.grad_h_s && a.ld_ghs < a.d_s) || (a.grad_w_s && a.ld_gws < a.d_s))
    return FCT_ERR_INVALID_ARG;
  if (!span_fits(a.BT, a.ld_hs, a.d_s, 2) || !span_fits(a.V, a.ld_ws, a.d_s, 2) ||
      !span_fits(a.BT, a.ld_ht, a.d_t, 2) || !span_fits(a.V, a.ld_wt, a.d_t, 2) ||
      (a.grad_h_s && !span_fits(a.BT, a.ld_ghs, a.d_s, 2)) ||
      (a.grad_w_s && !span_fits(a.V, a.ld_gws, a.d_s, 4)) || !span_fits(1, a.BT, a.BT, 8))
    return FCT_ERR_UNSUPPORTED;
  if (!a.h_s || !a.w_s || !a.h_t || !a.w_t || !a.target || !a.grad_ce || !a.grad_tvd)
    return FCT_ERR_INVALID_ARG;
  if (a.grad_stride != 0 && a.grad_stride != 1) return FCT_ERR_INVALID_ARG;
  const void* bf[5] = {a.h_s, a.w_s, a.h_t, a.w_t, a.grad_h_s};
  for (const void* q : bf)
    if (q && !aligned(q, 2)) return FCT_ERR_ALIGNMENT;
  if (!aligned(a.target, 8) || !aligned(a.grad_ce, 4) || !aligned(a.grad_tvd, 4) ||
      (a.grad_w_s && !aligned(a.grad_w_s, 4)) || (a.dev_status && !aligned(a.dev_status, 4)))
    return FCT_ERR_ALIGNMENT;
  float* outs[5] = {a.ce, a.tvd, a.lse_s, a.lse_t, a.sigma};
  Span outr[7];
  int n_out = 0;
  for (float* o : outs) {
    if (o == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(o, 4)) return FCT_ERR_ALIGNMENT;
    outr[n_out++] = mat_span(o, 1, a.BT, a.BT, 4);
  }
  if (a.grad_h_s) outr[n_out++] = mat_span(a.grad_h_s, a.BT, a.ld_ghs, a.d_s, 2);
  if (a.grad_w_s) outr[n_out++] = mat_span(a.grad_w_s, a.V, a.ld_gws, a.d_s, 4);
  const Span ins[4] = {mat_span(a.h_s, a.BT, a.ld_hs, a.d_s, 2),
                       mat_span(a.w_s, a.V, a.ld_ws, a.d_s, 2),
                       mat_span(a.h_t, a.BT, a.ld_ht, a.d_t, 2),
                       mat_span(a.w_t, a.V, a.ld_wt, a.d_t, 2)};
  for (int i = 0; i < n_out; ++i) {
    for (const Span& s : ins)
      if (overlap(outr[i], s)) return FCT_ERR_INVALID_ARG;
    for (int j = i + 1; j < n_out; ++j)
      if (overlap(outr[i], outr[j])) return FCT_ERR_INVALID_ARG;
  }
  return FCT_OK;
}

}  // namespace

extern "C" int fused_linear_ce_tvd_forward_backward_noalloc(
    const void* h_student, int64_t ld_h_student, const void* w_student, int64_t ld_w_student,
    int64_t d_student, const void* h_teacher, int64_t ld_h_teacher, const void* w_teacher,
    int64_t ld_w_teacher, int64_t d_teacher, const int64_t* target, int64_t BT, int64_t V,
    int64_t ignore_index, const float* grad_ce, const float* grad_tvd, int64_t grad_stride,
    float* ce, float* tvd, float* student_lse, float* teacher_lse, float* sigma,
    void* grad_h_student, int64_t ld_grad_h, float* grad_w_student, int64_t ld_grad_w,
    int32_t* dev_status, void* stream) {
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  if (BT == 0) return FCT_OK;
  fct::LinArgs a{h_student, ld_h_student, w_student, ld_w_student, d_student, h_teacher,
                 ld_h_teacher, w_teacher, ld_w_teacher, d_teacher, target, BT, V,
                 ignore_index, grad_ce, grad_tvd, grad_stride, ce, tvd, student_lse,
                 teacher_lse, sigma, grad_h_student, ld_grad_h, grad_w_student, ld_grad_w,
                 nullptr, 0, dev_status};
  int rc = check(a);
  if (rc != FCT_OK) return rc;
  // One student + one teacher fp32 row must fit in the scratch array.
  const size_t row_bytes = size_t(2) * sizeof(float) * size_t(fct::linear_logits_ld(V));
  if (row_bytes == 0 || row_bytes > kScratchBytes) return FCT_ERR_UNSUPPORTED;
  const int64_t per_block = static_cast<int64_t>(kScratchBytes / row_bytes);
  a.chunk_rows = per_block < BT ? per_block : BT;

  fct::FwdPlan plan;
  int device = 0, sms = 0;
  if ((rc = fct::plan_linear_forward(V, FCT_F32, &plan, &device, &sms)) != FCT_OK) return rc;
  if ((rc = scratch_on(device, &a.workspace)) != FCT_OK) return rc;
  if (run_blocks(a, plan, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FCT_ERR_CUDA;
  }
  return FCT_OK;
}
