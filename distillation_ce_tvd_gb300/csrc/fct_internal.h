// Internal launch interface between the C ABI (fct_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fused_ce_tvd.h"

namespace fct {

struct FwdArgs {
  const void* student;
  const void* teacher;  // unused by the plain cross-entropy forward
  int64_t ld_s, ld_t;
  int dtype;
  const int64_t* target;
  int64_t BT, V, ignore_index;
  float* ce;
  float* tvd;  // nullptr selects the plain cross-entropy forward
  float* lse_s;
  float* lse_t;
  float* sigma;
  int32_t* dev_status;
  // single-launch forward + backward only (nullptr grad: forward alone)
  void* grad;
  int64_t ld_g;
  const float* grad_ce;
  const float* grad_tvd;
  int64_t grad_stride;
  int keep_normal;  // 1: evict_normal instead of evict_last while a row must stay in L2
  int grad_bf16 = 0;  // single launch on fp32 logits: write the gradient as bf16
  // forward alone: per row, a uint32 tie flag then one byte of sign bits per
  // 16-byte vector (nullptr: none)
  uint8_t* signs = nullptr;
  int64_t ld_signs = 0;
  // start stagger (set by the launcher): cluster i of n waits stagger * i / n
  // clock cycles before its first load
  int64_t stagger = 0;
  // single launch with the row's log-sum-exp given as partials (the fused-
  // linear logits GEMM's epilogue writes them): per row lse_n base-2 states
  // (m2, s) at lse_part_s[row * lse_ld + j]; step 1 merges them instead of
  // reading the row (nullptr: step 1 reads the row)
  const float2* lse_part_s = nullptr;
  const float2* lse_part_t = nullptr;
  int64_t lse_ld = 0, lse_n = 0;
};

struct FwdPlan {
  bool vec;     // 16-byte vector path (pointers and strides aligned)
  int cluster;  // CTAs per row: 1, 2, 4 or 8
  int slots;    // rows in flight across the GPU (clusters launched), 0 = as many as fit
  bool keep_normal;  // L2 policy for rows that are read again (tuning)
  double stagger;    // start stagger, fraction of an estimated row time (0: none)
  int ring = 0;      // 0 automatic, 1 per-thread cp.async ring, 2 TMA bulk-copy ring
};

struct BwdArgs {
  const void* student;
  const void* teacher;  // nullptr selects the plain cross-entropy backward
  int64_t ld_s, ld_t;
  int dtype;
  const int64_t* target;
  int64_t BT, V, ignore_index;
  const float* lse_s;
  const float* lse_t;
  const float* sigma;
  const float* grad_ce;
  const float* grad_tvd;
  int64_t grad_stride;
  void* grad;
  int64_t ld_g;
  int32_t* dev_status;
  // the forward's sign words (see FwdArgs::signs), or nullptr
  const uint8_t* signs = nullptr;
  int64_t ld_signs = 0;
  // vocabulary shards: the logits are columns [tg_base, tg_base + V) of a
  // vocabulary of V_full entries (0: no shard).  Targets index the full
  // vocabulary; one outside this shard adds no -grad_ce term here, and only
  // one outside [0, V_full) is out of range.
  int64_t tg_base = 0;
  int64_t V_full = 0;
};

struct LossArgs {
  const int64_t* target;
  int64_t BT, ignore_index;
  const float* ce;   // nullptr: not summed
  const float* tvd;  // nullptr: not summed
  double alpha, beta;
  float* loss;       // outputs, each optional
  float* grad_ce;
  float* grad_tvd;
  int64_t* count;
};

// Fused-linear (hidden states and lm_head weights in, bf16) chunked loss.
struct LinArgs {
  const void* h_s;  // (BT, d_s) bf16
  int64_t ld_hs;
  const void* w_s;  // (V, d_s) bf16
  int64_t ld_ws, d_s;
  const void* h_t;  // (BT, d_t) bf16
  int64_t ld_ht;
  const void* w_t;  // (V, d_t) bf16
  int64_t ld_wt, d_t;
  const int64_t* target;
  int64_t BT, V, ignore_index;
  const float* grad_ce;
  const float* grad_tvd;
  int64_t grad_stride;
  float* ce;
  float* tvd;
  float* lse_s;
  float* lse_t;
  float* sigma;
  void* grad_h_s;   // (BT, d_s) bf16, or nullptr
  int64_t ld_ghs;
  float* grad_w_s;  // (V, d_s) fp32, accumulated, or nullptr
  int64_t ld_gws;
  void* workspace;  // linear_workspace_bytes(V, chunk_rows, logits_dtype), 256-byte aligned
  int64_t chunk_rows;
  int32_t* dev_status;
  int logits_dtype = FCT_F32;  // element type of the logit blocks
};

int64_t linear_logits_ld(int64_t V);
size_t linear_workspace_bytes(int64_t V, int64_t chunk_rows, int logits_dtype);
cudaError_t launch_linear(const LinArgs& a, const FwdPlan& plan, int device, int sms,
                          cudaStream_t st);

// The forward plan the fused-linear path uses (logit rows of width V and
// element type logits_dtype) on the calling thread's current device, with
// that device's index and SM count.  Returns an fct_status.
int plan_linear_forward(int64_t V, int logits_dtype, FwdPlan* plan, int* device, int* sms);

// Vocabulary shards (fct_vocab.cu): the passes over one shard's columns.
struct VpArgs {
  const void* student;  // the shard's first column of row 0
  const void* teacher;
  int64_t ld_s, ld_t;
  int dtype;
  const int64_t* target;  // indices into the full vocabulary
  int64_t BT, V;          // V: the shard's columns
  int64_t v_begin;        // the shard's first column in the full vocabulary
  int64_t ignore_index;
  const float* lse_s;     // pass 2: the merged lse values
  const float* lse_t;
  float* part;            // (BT, 3) after pass 1, (BT, 2) after pass 2
};

struct VpMergeArgs {
  const float* parts;  // (n_shards, BT, 3) or (n_shards, BT, 2)
  int64_t n_shards;
  const int64_t* target;
  int64_t BT, V;  // V: the full vocabulary
  int64_t ignore_index;
  float* ce;
  float* lse_s;
  float* lse_t;
  float* tvd;
  float* sigma;
  int32_t* dev_status;
};

cudaError_t launch_vp_pass(const VpArgs& a, bool vec, bool tvd_pass, int sms, cudaStream_t st);
cudaError_t launch_vp_merge(const VpMergeArgs& a, bool tvd_merge, cudaStream_t st);

// bf16 GEMM on the tensor cores (fct_gemm.cu): C(m, n) (+)= sum_k A(m, k) B(n, k).
// An operand is K-major (element (i, k) at ptr[i * ld + k]) or MN-major
// (element (i, k) at ptr[k * ld + i]); its base must be 16-byte aligned and
// ld a positive multiple of 8 (gemm_operand_ok).  c_kind: 0 fp32 C, 1 bf16
// C (rounded to nearest even), 2 fp32 C accumulated into.
struct GemmOperand {
  const void* ptr;
  int64_t ld;
  bool mn_major;
};
// split_ws (optional, 16-byte aligned): room for fp32 partial sums; a GEMM
// with too few output tiles to keep every SM pair busy and a long K may then
// split K (c_kind 0 and 1 only) and add the parts in a fixed order.
// gemm_split_workspace_bytes(M, N) is the most any split of an M x N result
// uses.
bool gemm_operand_ok(const void* p, int64_t ld);
// c_kind 3 (fp32 C) and 4 (bf16 C), both operands K-major only: also each
// row's base-2 log-sum-exp state (m2, s) over each 256-column tile t of C,
// at lse_part[row * lse_ld + t] (lse_ld >= the number of tiles), on the
// values as stored.
constexpr int kGemmLseTile = 256;
// Largest M, N or K: tile and box coordinates are 32-bit, and a tile's last
// rows (up to 1023 past its first) must not wrap.
constexpr int64_t kGemmMaxDim = (int64_t(1) << 31) - 1024;
cudaError_t launch_gemm(const GemmOperand& A, const GemmOperand& B, void* C, int64_t ldc,
                        int c_kind, int64_t M, int64_t N, int64_t K, int32_t* status, int sms,
                        cudaStream_t st, void* split_ws = nullptr, size_t split_ws_bytes = 0,
                        float2* lse_part = nullptr, int64_t lse_ld = 0);
size_t gemm_split_workspace_bytes(int64_t M, int64_t N);

cudaError_t launch_forward(const FwdArgs& a, const FwdPlan& plan, cudaStream_t st);
cudaError_t launch_mean(const LossArgs& a, cudaStream_t st);
cudaError_t launch_backward(const BwdArgs& a, bool vec, int sms, cudaStream_t st);

}  // namespace fct
