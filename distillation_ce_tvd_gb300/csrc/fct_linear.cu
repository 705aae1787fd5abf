// Fused-linear CE + TVD, chunked over rows.
//
// The loss of the PR #1384 analysis takes logits; a model produces them as
// hidden states times an lm_head weight.  Materialising the (BT, V) logits
// of student and teacher costs 2*BT*V elements of memory and traffic.  Here
// the rows go through in blocks of R: per block, two GEMMs (the library's
// tcgen05 GEMM, bf16 inputs, fp32 accumulate) write the block's student and
// teacher logits into the caller's workspace, the single-launch forward +
// backward kernel reads them and writes the block's logit gradient as bf16,
// and two more GEMMs give the block's d loss / d hidden and accumulate
// d loss / d weight (their transposed operands are read in place, as
// MN-major tiles).  The logit blocks are fp32 (the GEMMs' own precision), or
// bf16 (rounded once by the GEMM, as a model's bf16 lm_head produces them),
// which halves their bytes and lets the gradient overwrite the student block
// in place.  The logits GEMMs' epilogue also folds each row's values into
// base-2 log-sum-exp states per 256-column tile, so the loss kernel merges
// those instead of reading the block for its step 1: two passes over the
// block instead of three, and only the student stays in L2 between them.  Only the block's logits and gradient exist at a time.  The
// teacher is frozen (no gradients).
#include <cstdint>

#include "fct_common.cuh"
#include "fct_internal.h"

namespace fct {

int64_t linear_logits_ld(int64_t V) { return (V + 7) / 8 * 8; }

// Log-sum-exp partial states per logit row: one per 256-column tile.
int64_t linear_lse_parts(int64_t V) { return (V + kGemmLseTile - 1) / kGemmLseTile; }

size_t linear_workspace_bytes(int64_t V, int64_t chunk_rows, int logits_dtype) {
  // bf16: two student blocks (the logit gradient is written over the
  // student's, and d weight takes two blocks' gradients at once) and the
  // teacher block; fp32: the student and teacher blocks, then two bf16
  // logit-gradient blocks; then the student's and the teacher's
  // log-sum-exp partials
  // SIZE_MAX when the size does not fit a size_t (no workspace can hold it)
  const uint64_t per_entry = logits_dtype == FCT_BF16 ? 3 * sizeof(uint16_t)
                                                      : 2 * sizeof(float) + 2 * sizeof(uint16_t);
  const uint64_t rows = uint64_t(chunk_rows);
  const uint64_t row_bytes = uint64_t(linear_logits_ld(V)) * per_entry +
                             2 * uint64_t(linear_lse_parts(V)) * sizeof(float2);
  if (chunk_rows <= 0 || V <= 0 || row_bytes > SIZE_MAX / rows) return SIZE_MAX;
  return size_t(rows * row_bytes);
}

cudaError_t launch_linear(const LinArgs& a, const FwdPlan& plan, int device, int sms,
                          cudaStream_t st) {
  (void)device;
  // logit rows padded to a multiple of 8 elements: 16-byte (bf16) or 32-byte
  // (fp32) row strides, so the loss kernel's vector path applies
  const int64_t ldl = linear_logits_ld(a.V);
  const bool bf16 = a.logits_dtype == FCT_BF16;
  const int64_t block_bytes = a.chunk_rows * ldl * (bf16 ? 2 : 4);
  const int64_t gblock = a.chunk_rows * ldl;  // elements of one bf16 gradient block
  char* base = static_cast<char*>(a.workspace);
  // bf16: student blocks 0 and 1 (block b uses b % 2; its gradient goes over
  // it), then the teacher block; fp32: student, teacher, gradient blocks 0, 1
  char* Lt = base + (bf16 ? 2 : 1) * block_bytes;
  uint16_t* G0 = bf16 ? reinterpret_cast<uint16_t*>(base)
                      : reinterpret_cast<uint16_t*>(Lt + block_bytes);
  const int64_t ldg = ldl;
  // the logits GEMMs also write each row's log-sum-exp partials, so the loss
  // kernel starts at step 2
  const int lkind = bf16 ? 4 : 3;
  const int64_t n_parts = linear_lse_parts(a.V);
  float2* Ps = reinterpret_cast<float2*>(bf16 ? Lt + block_bytes
                                              : reinterpret_cast<char*>(G0 + 2 * gblock));
  float2* Pt = Ps + a.chunk_rows * n_parts;
  const auto* Hs = static_cast<const uint16_t*>(a.h_s);
  const auto* Ht = static_cast<const uint16_t*>(a.h_t);
  const GemmOperand Ws{a.w_s, a.ld_ws, false}, Wt{a.w_t, a.ld_wt, false};
  cudaError_t e;

  int64_t b = 0;
  for (int64_t r0 = 0; r0 < a.BT; r0 += a.chunk_rows, ++b) {
    const int64_t R = (a.BT - r0 < a.chunk_rows) ? a.BT - r0 : a.chunk_rows;
    uint16_t* G = G0 + (b & 1) * gblock;  // this block's logit gradient
    void* Ls = bf16 ? static_cast<void*>(G) : static_cast<void*>(base);
    // logits (R x V) = H (R x D) W^T: both operands K-major
    const GemmOperand Hsb{Hs + r0 * a.ld_hs, a.ld_hs, false}, Htb{Ht + r0 * a.ld_ht, a.ld_ht, false};
    if ((e = launch_gemm(Hsb, Ws, Ls, ldl, lkind, R, a.V, a.d_s, a.dev_status, sms, st, nullptr,
                         0, Ps, n_parts)) != cudaSuccess)
      return e;
    if ((e = launch_gemm(Htb, Wt, Lt, ldl, lkind, R, a.V, a.d_t, a.dev_status, sms, st, nullptr,
                         0, Pt, n_parts)) != cudaSuccess)
      return e;
    // the loss on the block; its logit gradient, as bf16, into G
    FwdArgs f{Ls, Lt, ldl, ldl, bf16 ? FCT_BF16 : FCT_F32, a.target + r0, R, a.V, a.ignore_index,
              a.ce + r0, a.tvd + r0, a.lse_s + r0, a.lse_t + r0, a.sigma + r0, a.dev_status,
              G, ldg, a.grad_ce + (a.grad_stride ? r0 : 0),
              a.grad_tvd + (a.grad_stride ? r0 : 0), a.grad_stride, plan.keep_normal ? 1 : 0,
              /*grad_bf16=*/bf16 ? 0 : 1};
    f.lse_part_s = Ps;
    f.lse_part_t = Pt;
    f.lse_ld = n_parts;
    f.lse_n = n_parts;
    if ((e = launch_forward(f, plan, st)) != cudaSuccess) return e;
    if (a.grad_h_s == nullptr && a.grad_w_s == nullptr) continue;
    // d hidden (R x D, bf16) = G (R x V) W (V x D): C(r, d) = sum_v G(r, v) W(v, d),
    // G K-major, W read as the MN-major (D x V) operand.  Few output tiles
    // and a K of V: the GEMM may split K, with its partial sums in the
    // teacher block, which the loss kernel has finished reading.
    if (a.grad_h_s &&
        (e = launch_gemm(GemmOperand{G, ldg, false}, GemmOperand{a.w_s, a.ld_ws, true},
                         static_cast<uint16_t*>(a.grad_h_s) + r0 * a.ld_ghs, a.ld_ghs,
                         FCT_GEMM_BF16, R, a.d_s, a.V, a.dev_status, sms, st, Lt,
                         size_t(block_bytes))) != cudaSuccess)
      return e;
    // d weight (V x D, fp32) += G^T H: C(v, d) += sum_r G(r, v) H(r, d), both
    // operands MN-major, once per two blocks (K = their rows, the gradient
    // blocks adjacent in the workspace), or for a last block left alone:
    // one read-modify-write of the fp32 (V, D) gradient per two blocks
    const bool last = r0 + R >= a.BT;
    if (a.grad_w_s && ((b & 1) || last)) {
      const int64_t k0 = (b & 1) ? r0 - a.chunk_rows : r0;  // first row of the pending blocks
      if ((e = launch_gemm(GemmOperand{G0, ldg, true},
                           GemmOperand{Hs + k0 * a.ld_hs, a.ld_hs, true}, a.grad_w_s, a.ld_gws,
                           FCT_GEMM_ADD_F32, a.V, a.d_s, r0 + R - k0, a.dev_status, sms, st)) !=
          cudaSuccess)
        return e;
    }
  }
  return cudaGetLastError();
}

}  // namespace fct
