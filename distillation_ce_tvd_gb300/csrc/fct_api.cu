// C ABI of libfused_ce_tvd.so: argument checks, launch planning, dispatch.
// The operations themselves are described in include/fused_ce_tvd.h.
#include <mutex>

#include "fct_internal.h"

namespace {

struct DeviceInfo {
  int sms = 0;
  int l2_bytes = 0;
  int major = 0, minor = 0;
  bool ok = false;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

// Properties of the calling thread's current device, queried once.
int current_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FCT_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return FCT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ok) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return FCT_ERR_CUDA;
    }
    d.ok = true;
  }
  *out = d;
  // The kernels are built for sm_103a only.
  if (d.major != 10 || d.minor != 3) return FCT_ERR_UNSUPPORTED;
  return FCT_OK;
}

size_t elem_size(int dtype) { return dtype == FCT_BF16 ? 2 : 4; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte range [lo, hi) covered by a (rows, cols) matrix with row stride ld.
struct Range {
  uintptr_t lo, hi;
};
Range mat_range(const void* p, int64_t rows, int64_t ld, int64_t cols, size_t e) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * static_cast<int64_t>(e))};
}
Range vec_range(const void* p, int64_t n, size_t e) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + static_cast<uintptr_t>(n * static_cast<int64_t>(e))};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// Whether a (rows, cols) matrix of e-byte elements with row stride ld spans
// at most 2^62 bytes, checked without overflowing, so that every byte range
// and element offset computed from the sizes is exact.
bool span_fits(int64_t rows, int64_t ld, int64_t cols, int64_t e) {
  const int64_t lim = (int64_t(1) << 62) / e;
  if (rows <= 0 || cols <= 0 || ld < cols || cols > lim) return false;
  return rows - 1 <= (lim - cols) / ld;
}

int check_logits(const void* x, int64_t ld, int dtype, int64_t V, int64_t BT) {
  if (x == nullptr) return FCT_ERR_INVALID_ARG;
  if (ld < V) return FCT_ERR_INVALID_ARG;
  if (!span_fits(BT, ld, V, static_cast<int64_t>(elem_size(dtype)))) return FCT_ERR_UNSUPPORTED;
  if (!aligned(x, elem_size(dtype))) return FCT_ERR_ALIGNMENT;
  return FCT_OK;
}

// Sign words of one row: a uint32 tie flag, then one byte per 16-byte vector
// (the row's ragged tail has none), padded to a multiple of 4 bytes.
int64_t signs_row_bytes(int64_t V, int dtype) {
  const int64_t nvec = V / (16 / static_cast<int64_t>(elem_size(dtype)));
  return 4 + (nvec + 3) / 4 * 4;
}

bool vec_ok(const void* x, int64_t ld, int dtype) {
  return aligned(x, 16) && ((ld * static_cast<int64_t>(elem_size(dtype))) % 16) == 0;
}

int check_common(int dtype, const int64_t* target, int64_t BT, int64_t V) {
  if (dtype != FCT_F32 && dtype != FCT_BF16) return FCT_ERR_UNSUPPORTED;
  if (V <= 0) return FCT_ERR_INVALID_ARG;
  if (target == nullptr) return FCT_ERR_INVALID_ARG;
  if (!aligned(target, 8)) return FCT_ERR_ALIGNMENT;
  (void)BT;
  return FCT_OK;
}

// Launch options of one call: NULL means automatic.  Returns an fct_status.
int check_options(const fct_options* o) {
  if (o == nullptr) return FCT_OK;
  const int c = o->ctas_per_row;
  if (c != 0 && c != 1 && c != 2 && c != 4 && c != 8) return FCT_ERR_INVALID_ARG;
  if (o->l2_keep != 0 && o->l2_keep != 1) return FCT_ERR_INVALID_ARG;
  if (!(o->stagger <= 4.0f)) return FCT_ERR_INVALID_ARG;  // rejects NaN too
  if (o->ring < 0 || o->ring > 2) return FCT_ERR_INVALID_ARG;
  for (int32_t r : o->reserved)
    if (r != 0) return FCT_ERR_INVALID_ARG;
  return FCT_OK;
}

// Default start stagger of the multi-pass forward kernels: half of an
// estimated row time (measured best for the forward alone, inside the flat
// optimum for the single launch at 8192 x 151936 bf16).
constexpr double kDefaultStagger = 0.5;

// Rows in flight and CTAs per row for the multi-pass forward kernels.  A
// later pass re-reads each row from L2, so the rows in flight times the
// bytes of the kept row should stay near the L2 size; rows are split over a
// cluster of C CTAs until every SM still gets at least one CTA.  The kept
// row is student + teacher for the fused loss (tvd), the student alone for
// cross-entropy in one launch (ce_grad), or kept_rows rows when given (the
// fused-linear loss starts from given states and re-reads only the student).
// Budget: 1.10 of L2 for the fused loss (measured on GB300 with staggered
// CTAs, single launch and forward alone: one CTA per row on the bulk-copy
// ring beats 2-CTA clusters up to 960 KB of student + teacher row, bf16
// V = 240000 and fp32 V = 121000, by up to 30%, and loses at 1.02 MB; the
// rows in flight are in different passes, the first one's row still
// arriving and the third one's shrinking); 0.80 for cross-entropy alone
// (its single launch measured faster on 2-CTA clusters than at one CTA per
// row for student rows of 760 to 980 KB, fp32 and bf16).
// Depends on V, the element type, the device and the call's options only
// (never on BT), so results do not depend on how the rows are batched.
fct::FwdPlan plan_forward(const DeviceInfo& d, int64_t V, int dtype, bool tvd, bool vec,
                          bool ce_grad = false, const fct_options* opts = nullptr,
                          int kept_rows = 0) {
  fct::FwdPlan plan{vec, 1, 0, false, kDefaultStagger, 0};
  if (opts != nullptr) {
    plan.ring = opts->ring;
    plan.keep_normal = opts->l2_keep == 1;
    if (opts->stagger > 0.f) plan.stagger = opts->stagger;
    if (opts->stagger < 0.f) plan.stagger = 0.0;
  }
  if (!tvd && !ce_grad) return plan;  // one pass: nothing to keep in L2
  const double rows_kept = kept_rows > 0 ? double(kept_rows) : (tvd ? 2.0 : 1.0);
  const double row_bytes = rows_kept * static_cast<double>(V) * static_cast<double>(elem_size(dtype));
  const double budget = (tvd ? 1.10 : 0.80) * static_cast<double>(d.l2_bytes);
  int64_t fit = static_cast<int64_t>(budget / row_bytes);
  if (fit < 1) fit = 1;
  int C = opts ? opts->ctas_per_row : 0;
  if (C == 0) {
    C = 1;
    while (C < 8 && fit * C < d.sms) C *= 2;
  }
  int64_t per_sm = (fit * C) / d.sms;
  if (per_sm < 1) per_sm = 1;
  if (per_sm > 4) per_sm = 4;
  plan.cluster = C;
  plan.slots = static_cast<int>((d.sms * per_sm) / C);
  if (plan.slots < 1) plan.slots = 1;
  return plan;
}

int forward_impl(const void* student, int64_t ld_s, const void* teacher, int64_t ld_t,
                 int dtype, const int64_t* target, int64_t BT, int64_t V, int64_t ignore_index,
                 float* ce, float* tvd, float* lse_s, float* lse_t, float* sigma,
                 int32_t* dev_status, void* stream, uint8_t* signs = nullptr,
                 int64_t ld_signs = 0, const fct_options* opts = nullptr) {
  const bool fused = (tvd != nullptr);
  if (signs != nullptr && !fused) return FCT_ERR_INVALID_ARG;
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  int rc = check_options(opts);
  if (rc != FCT_OK) return rc;
  if (BT == 0) return FCT_OK;
  rc = check_common(dtype, target, BT, V);
  if (rc != FCT_OK) return rc;
  if ((rc = check_logits(student, ld_s, dtype, V, BT)) != FCT_OK) return rc;
  if (fused && (rc = check_logits(teacher, ld_t, dtype, V, BT)) != FCT_OK) return rc;
  float* outs[5] = {ce, lse_s, tvd, lse_t, sigma};
  const int n_out = fused ? 5 : 2;
  for (int i = 0; i < n_out; ++i) {
    if (outs[i] == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(outs[i], 4)) return FCT_ERR_ALIGNMENT;
  }
  if (dev_status && !aligned(dev_status, 4)) return FCT_ERR_ALIGNMENT;
  const size_t e = elem_size(dtype);
  Range ins[3] = {mat_range(student, BT, ld_s, V, e),
                  fused ? mat_range(teacher, BT, ld_t, V, e) : Range{0, 0},
                  vec_range(target, BT, 8)};
  for (int i = 0; i < n_out; ++i) {
    const Range r = vec_range(outs[i], BT, 4);
    for (int j = 0; j < 3; ++j)
      if (overlap(r, ins[j])) return FCT_ERR_INVALID_ARG;
    for (int j = i + 1; j < n_out; ++j)
      if (overlap(r, vec_range(outs[j], BT, 4))) return FCT_ERR_INVALID_ARG;
  }
  const int64_t sb = signs_row_bytes(V, dtype);
  if (signs != nullptr) {
    if (!aligned(signs, 4) || ld_signs % 4 != 0) return FCT_ERR_ALIGNMENT;
    if (ld_signs < sb) return FCT_ERR_INVALID_ARG;
    const Range r = mat_range(signs, BT, ld_signs, sb, 1);
    for (int j = 0; j < 3; ++j)
      if (overlap(r, ins[j])) return FCT_ERR_INVALID_ARG;
    for (int i = 0; i < n_out; ++i)
      if (overlap(r, vec_range(outs[i], BT, 4))) return FCT_ERR_INVALID_ARG;
  }

  DeviceInfo d;
  if ((rc = current_device(&d)) != FCT_OK) return rc;
  const bool vec = vec_ok(student, ld_s, dtype) && (!fused || vec_ok(teacher, ld_t, dtype));
  fct::FwdArgs a{student, teacher, ld_s, ld_t, dtype, target, BT, V, ignore_index,
                 ce, tvd, lse_s, lse_t, sigma, dev_status, nullptr, 0, nullptr, nullptr, 0, 0};
  // Cross-entropy alone takes the row split of its single launch
  // (ce_forward_backward), so both reduce each row in the same order and give
  // the same bits.
  const fct::FwdPlan plan = plan_forward(d, V, dtype, fused, vec, /*ce_grad=*/!fused, opts);
  a.keep_normal = plan.keep_normal ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (signs != nullptr) {
    if (vec) {
      a.signs = signs;
      a.ld_signs = ld_signs;
    } else if (cudaMemset2DAsync(signs, static_cast<size_t>(ld_signs), 0x01, 4,
                                 static_cast<size_t>(BT), st) != cudaSuccess) {
      // unaligned rows have no sign words: every row's tie flag is set, so
      // the backward recomputes the signs from the teacher
      cudaGetLastError();
      return FCT_ERR_CUDA;
    }
  }
  if (fct::launch_forward(a, plan, st) != cudaSuccess) return FCT_ERR_CUDA;
  return FCT_OK;
}

int backward_impl(const void* student, int64_t ld_s, const void* teacher, int64_t ld_t,
                  int dtype, const int64_t* target, int64_t BT, int64_t V, int64_t ignore_index,
                  const float* lse_s, const float* lse_t, const float* sigma,
                  const float* grad_ce, const float* grad_tvd, int64_t grad_stride,
                  void* grad, int64_t ld_g, int32_t* dev_status, void* stream,
                  const uint8_t* signs = nullptr, int64_t ld_signs = 0, int64_t tg_base = 0,
                  int64_t V_full = 0) {
  const bool fused = (teacher != nullptr) || (lse_t != nullptr);
  if (signs != nullptr && !fused) return FCT_ERR_INVALID_ARG;
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  if (BT == 0) return FCT_OK;
  int rc = check_common(dtype, target, BT, V);
  if (rc != FCT_OK) return rc;
  if ((rc = check_logits(student, ld_s, dtype, V, BT)) != FCT_OK) return rc;
  if (fused && (rc = check_logits(teacher, ld_t, dtype, V, BT)) != FCT_OK) return rc;
  if ((rc = check_logits(grad, ld_g, dtype, V, BT)) != FCT_OK) return rc;
  if (grad_stride != 0 && grad_stride != 1) return FCT_ERR_INVALID_ARG;
  const float* rows[5] = {lse_s, grad_ce, lse_t, sigma, grad_tvd};
  const int n_rows = fused ? 5 : 2;
  for (int i = 0; i < n_rows; ++i) {
    if (rows[i] == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(rows[i], 4)) return FCT_ERR_ALIGNMENT;
  }
  if (dev_status && !aligned(dev_status, 4)) return FCT_ERR_ALIGNMENT;
  const size_t e = elem_size(dtype);
  const Range g = mat_range(grad, BT, ld_g, V, e);
  const bool inplace = (grad == student);
  if (inplace && ld_g != ld_s) return FCT_ERR_INVALID_ARG;
  if (!inplace && overlap(g, mat_range(student, BT, ld_s, V, e))) return FCT_ERR_INVALID_ARG;
  if (fused && overlap(g, mat_range(teacher, BT, ld_t, V, e))) return FCT_ERR_INVALID_ARG;
  if (overlap(g, vec_range(target, BT, 8))) return FCT_ERR_INVALID_ARG;
  for (int i = 0; i < n_rows; ++i) {
    const int64_t n = (i == 1 || i == 4) ? (grad_stride ? BT : 1) : BT;
    if (overlap(g, vec_range(rows[i], n, 4))) return FCT_ERR_INVALID_ARG;
  }
  if (signs != nullptr) {
    if (!aligned(signs, 4) || ld_signs % 4 != 0) return FCT_ERR_ALIGNMENT;
    if (ld_signs < signs_row_bytes(V, dtype)) return FCT_ERR_INVALID_ARG;
    if (overlap(g, mat_range(signs, BT, ld_signs, signs_row_bytes(V, dtype), 1)))
      return FCT_ERR_INVALID_ARG;
  }

  DeviceInfo d;
  if ((rc = current_device(&d)) != FCT_OK) return rc;
  const bool vec = vec_ok(student, ld_s, dtype) && vec_ok(grad, ld_g, dtype) &&
                   (!fused || vec_ok(teacher, ld_t, dtype));
  fct::BwdArgs a{student, fused ? teacher : nullptr, ld_s, ld_t, dtype, target, BT, V,
                 ignore_index, lse_s, lse_t, sigma, grad_ce, grad_tvd, grad_stride,
                 grad, ld_g, dev_status};
  if (signs != nullptr && vec) {  // without the vector path the signs are recomputed
    a.signs = signs;
    a.ld_signs = ld_signs;
  }
  a.tg_base = tg_base;
  a.V_full = V_full;
  if (fct::launch_backward(a, vec, d.sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

// Single-launch forward + backward: the checks of both calls, plus no
// overlap between the gradient and the per-row outputs.
int forward_backward_impl(const void* student, int64_t ld_s, const void* teacher, int64_t ld_t,
                          int dtype, const int64_t* target, int64_t BT, int64_t V,
                          int64_t ignore_index, const float* grad_ce, const float* grad_tvd,
                          int64_t grad_stride, float* ce, float* tvd, float* lse_s, float* lse_t,
                          float* sigma, void* grad, int64_t ld_g, int32_t* dev_status,
                          void* stream, const fct_options* opts = nullptr) {
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  int rc = check_options(opts);
  if (rc != FCT_OK) return rc;
  if (BT == 0) return FCT_OK;
  rc = check_common(dtype, target, BT, V);
  if (rc != FCT_OK) return rc;
  if ((rc = check_logits(student, ld_s, dtype, V, BT)) != FCT_OK) return rc;
  if ((rc = check_logits(teacher, ld_t, dtype, V, BT)) != FCT_OK) return rc;
  if ((rc = check_logits(grad, ld_g, dtype, V, BT)) != FCT_OK) return rc;
  if (grad_stride != 0 && grad_stride != 1) return FCT_ERR_INVALID_ARG;
  if (grad_ce == nullptr || grad_tvd == nullptr) return FCT_ERR_INVALID_ARG;
  if (!aligned(grad_ce, 4) || !aligned(grad_tvd, 4)) return FCT_ERR_ALIGNMENT;
  float* outs[5] = {ce, tvd, lse_s, lse_t, sigma};
  for (int i = 0; i < 5; ++i) {
    if (outs[i] == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(outs[i], 4)) return FCT_ERR_ALIGNMENT;
  }
  if (dev_status && !aligned(dev_status, 4)) return FCT_ERR_ALIGNMENT;
  const size_t e = elem_size(dtype);
  const Range rs = mat_range(student, BT, ld_s, V, e), rt = mat_range(teacher, BT, ld_t, V, e);
  const Range rtg = vec_range(target, BT, 8), g = mat_range(grad, BT, ld_g, V, e);
  const int64_t n_up = grad_stride ? BT : 1;
  const Range rgc = vec_range(grad_ce, n_up, 4), rgt = vec_range(grad_tvd, n_up, 4);
  const bool inplace = (grad == student);
  if (inplace && ld_g != ld_s) return FCT_ERR_INVALID_ARG;
  if (!inplace && overlap(g, rs)) return FCT_ERR_INVALID_ARG;
  if (overlap(g, rt) || overlap(g, rtg) || overlap(g, rgc) || overlap(g, rgt))
    return FCT_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i) {
    const Range r = vec_range(outs[i], BT, 4);
    if (overlap(r, rs) || overlap(r, rt) || overlap(r, rtg) || overlap(r, g) ||
        overlap(r, rgc) || overlap(r, rgt))
      return FCT_ERR_INVALID_ARG;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(r, vec_range(outs[j], BT, 4))) return FCT_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  if ((rc = current_device(&d)) != FCT_OK) return rc;
  const bool vec = vec_ok(student, ld_s, dtype) && vec_ok(teacher, ld_t, dtype) &&
                   vec_ok(grad, ld_g, dtype);
  if (!vec) {
    // Unaligned rows: the two-launch path gives the same results.
    rc = forward_impl(student, ld_s, teacher, ld_t, dtype, target, BT, V, ignore_index, ce, tvd,
                      lse_s, lse_t, sigma, dev_status, stream, nullptr, 0, opts);
    if (rc != FCT_OK) return rc;
    return backward_impl(student, ld_s, teacher, ld_t, dtype, target, BT, V, ignore_index, lse_s,
                         lse_t, sigma, grad_ce, grad_tvd, grad_stride, grad, ld_g, dev_status,
                         stream);
  }
  fct::FwdArgs a{student, teacher, ld_s, ld_t, dtype, target, BT, V, ignore_index,
                 ce, tvd, lse_s, lse_t, sigma, dev_status, grad, ld_g, grad_ce, grad_tvd,
                 grad_stride, 0};
  const fct::FwdPlan plan = plan_forward(d, V, dtype, true, true, false, opts);
  a.keep_normal = plan.keep_normal ? 1 : 0;
  if (fct::launch_forward(a, plan, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

// Cross-entropy forward + backward in one launch: ce_forward's and
// ce_backward's checks, no overlap between the gradient and the per-row
// outputs; unaligned rows take the two launches (same results).
int ce_forward_backward_impl(const void* logits, int64_t ld, int dtype, const int64_t* target,
                             int64_t BT, int64_t V, int64_t ignore_index, const float* grad_ce,
                             int64_t grad_stride, float* ce, float* lse, void* grad, int64_t ld_g,
                             int32_t* dev_status, void* stream, const fct_options* opts = nullptr) {
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  int rc = check_options(opts);
  if (rc != FCT_OK) return rc;
  if (BT == 0) return FCT_OK;
  rc = check_common(dtype, target, BT, V);
  if (rc != FCT_OK) return rc;
  if ((rc = check_logits(logits, ld, dtype, V, BT)) != FCT_OK) return rc;
  if ((rc = check_logits(grad, ld_g, dtype, V, BT)) != FCT_OK) return rc;
  if (grad_stride != 0 && grad_stride != 1) return FCT_ERR_INVALID_ARG;
  if (grad_ce == nullptr || ce == nullptr || lse == nullptr) return FCT_ERR_INVALID_ARG;
  if (!aligned(grad_ce, 4) || !aligned(ce, 4) || !aligned(lse, 4)) return FCT_ERR_ALIGNMENT;
  if (dev_status && !aligned(dev_status, 4)) return FCT_ERR_ALIGNMENT;
  const size_t e = elem_size(dtype);
  const Range rs = mat_range(logits, BT, ld, V, e), g = mat_range(grad, BT, ld_g, V, e);
  const Range rtg = vec_range(target, BT, 8), rgc = vec_range(grad_ce, grad_stride ? BT : 1, 4);
  const bool inplace = (grad == logits);
  if (inplace && ld_g != ld) return FCT_ERR_INVALID_ARG;
  if (!inplace && overlap(g, rs)) return FCT_ERR_INVALID_ARG;
  if (overlap(g, rtg) || overlap(g, rgc)) return FCT_ERR_INVALID_ARG;
  const Range rce = vec_range(ce, BT, 4), rl = vec_range(lse, BT, 4);
  if (overlap(rce, rl)) return FCT_ERR_INVALID_ARG;
  for (const Range& r : {rce, rl})
    if (overlap(r, rs) || overlap(r, rtg) || overlap(r, g) || overlap(r, rgc))
      return FCT_ERR_INVALID_ARG;
  DeviceInfo d;
  if ((rc = current_device(&d)) != FCT_OK) return rc;
  if (!(vec_ok(logits, ld, dtype) && vec_ok(grad, ld_g, dtype))) {
    rc = forward_impl(logits, ld, nullptr, ld, dtype, target, BT, V, ignore_index, ce, nullptr,
                      lse, nullptr, nullptr, dev_status, stream, nullptr, 0, opts);
    if (rc != FCT_OK) return rc;
    return backward_impl(logits, ld, nullptr, ld, dtype, target, BT, V, ignore_index, lse,
                         nullptr, nullptr, grad_ce, nullptr, grad_stride, grad, ld_g, dev_status,
                         stream);
  }
  fct::FwdArgs a{logits, nullptr, ld, ld, dtype, target, BT, V, ignore_index,
                 ce, nullptr, lse, nullptr, nullptr, dev_status, grad, ld_g, grad_ce, nullptr,
                 grad_stride, 0};
  const fct::FwdPlan plan = plan_forward(d, V, dtype, false, true, /*ce_grad=*/true, opts);
  a.keep_normal = plan.keep_normal ? 1 : 0;
  if (fct::launch_forward(a, plan, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

int linear_impl(const void* h_s, int64_t ld_hs, const void* w_s, int64_t ld_ws, int64_t d_s,
                const void* h_t, int64_t ld_ht, const void* w_t, int64_t ld_wt, int64_t d_t,
                const int64_t* target, int64_t BT, int64_t V, int64_t ignore_index,
                const float* grad_ce, const float* grad_tvd, int64_t grad_stride, float* ce,
                float* tvd, float* lse_s, float* lse_t, float* sigma, void* grad_h_s,
                int64_t ld_ghs, float* grad_w_s, int64_t ld_gws, int logits_dtype,
                void* workspace, size_t workspace_bytes, int64_t chunk_rows,
                int32_t* dev_status, void* stream) {
  if (BT < 0 || V <= 0 || d_s <= 0 || d_t <= 0 || chunk_rows <= 0) return FCT_ERR_INVALID_ARG;
  if (logits_dtype != FCT_F32 && logits_dtype != FCT_BF16) return FCT_ERR_UNSUPPORTED;
  if (BT == 0) return FCT_OK;
  if (ld_hs < d_s || ld_ws < d_s || ld_ht < d_t || ld_wt < d_t) return FCT_ERR_INVALID_ARG;
  if ((grad_h_s && ld_ghs < d_s) || (grad_w_s && ld_gws < d_s)) return FCT_ERR_INVALID_ARG;
  if (!span_fits(BT, ld_hs, d_s, 2) || !span_fits(V, ld_ws, d_s, 2) ||
      !span_fits(BT, ld_ht, d_t, 2) || !span_fits(V, ld_wt, d_t, 2) ||
      (grad_h_s && !span_fits(BT, ld_ghs, d_s, 2)) ||
      (grad_w_s && !span_fits(V, ld_gws, d_s, 4)) || !span_fits(1, BT, BT, 8))
    return FCT_ERR_UNSUPPORTED;
  // the GEMMs' dimensions (V, d, and up to two row blocks as K) within the
  // range of their 32-bit tile coordinates
  const int64_t kDim = fct::kGemmMaxDim;
  if (V > kDim || d_s > kDim || d_t > kDim || ld_hs > kDim || ld_ws > kDim || ld_ht > kDim ||
      ld_wt > kDim || ld_ghs > kDim || ld_gws > kDim || chunk_rows > kDim / 2)
    return FCT_ERR_UNSUPPORTED;
  if (!h_s || !w_s || !h_t || !w_t || !target || !grad_ce || !grad_tvd || !workspace)
    return FCT_ERR_INVALID_ARG;
  if (ld_hs < d_s || ld_ws < d_s || ld_ht < d_t || ld_wt < d_t) return FCT_ERR_INVALID_ARG;
  if (grad_h_s && ld_ghs < d_s) return FCT_ERR_INVALID_ARG;
  if (grad_w_s && ld_gws < d_s) return FCT_ERR_INVALID_ARG;
  if (grad_stride != 0 && grad_stride != 1) return FCT_ERR_INVALID_ARG;
  // the GEMM operands are TMA tiles: 16-byte aligned rows
  if (!fct::gemm_operand_ok(h_s, ld_hs) || !fct::gemm_operand_ok(w_s, ld_ws) ||
      !fct::gemm_operand_ok(h_t, ld_ht) || !fct::gemm_operand_ok(w_t, ld_wt) ||
      (grad_h_s && !aligned(grad_h_s, 2)))
    return FCT_ERR_ALIGNMENT;
  if (!aligned(target, 8) || !aligned(grad_ce, 4) || !aligned(grad_tvd, 4) ||
      (grad_w_s && !aligned(grad_w_s, 4)) || !aligned(workspace, 256) ||
      (dev_status && !aligned(dev_status, 4)))
    return FCT_ERR_ALIGNMENT;
  float* outs[5] = {ce, tvd, lse_s, lse_t, sigma};
  for (int i = 0; i < 5; ++i) {
    if (outs[i] == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(outs[i], 4)) return FCT_ERR_ALIGNMENT;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(vec_range(outs[i], BT, 4), vec_range(outs[j], BT, 4))) return FCT_ERR_INVALID_ARG;
  }
  const int64_t rows = chunk_rows < BT ? chunk_rows : BT;
  if (workspace_bytes < fct::linear_workspace_bytes(V, rows, logits_dtype))
    return FCT_ERR_INVALID_ARG;
  // outputs must not overlap the inputs or the workspace
  const Range ins[5] = {mat_range(h_s, BT, ld_hs, d_s, 2), mat_range(w_s, V, ld_ws, d_s, 2),
                        mat_range(h_t, BT, ld_ht, d_t, 2), mat_range(w_t, V, ld_wt, d_t, 2),
                        vec_range(workspace, static_cast<int64_t>(workspace_bytes), 1)};
  Range outr[7];
  int n_out = 0;
  for (int i = 0; i < 5; ++i) outr[n_out++] = vec_range(outs[i], BT, 4);
  if (grad_h_s) outr[n_out++] = mat_range(grad_h_s, BT, ld_ghs, d_s, 2);
  if (grad_w_s) outr[n_out++] = mat_range(grad_w_s, V, ld_gws, d_s, 4);
  for (int i = 0; i < n_out; ++i)
    for (int j = 0; j < 5; ++j)
      if (overlap(outr[i], ins[j])) return FCT_ERR_INVALID_ARG;
  if (grad_h_s && grad_w_s && overlap(outr[5], outr[6])) return FCT_ERR_INVALID_ARG;

  DeviceInfo d;
  int rc = current_device(&d);
  if (rc != FCT_OK) return rc;
  int dev = 0;
  cudaGetDevice(&dev);
  fct::LinArgs a{h_s, ld_hs, w_s, ld_ws, d_s, h_t, ld_ht, w_t, ld_wt, d_t, target, BT, V,
                 ignore_index, grad_ce, grad_tvd, grad_stride, ce, tvd, lse_s, lse_t, sigma,
                 grad_h_s, ld_ghs, grad_w_s, ld_gws, workspace, chunk_rows, dev_status,
                 logits_dtype};
  // the loss kernel starts from the logits GEMMs' states: only the student
  // block's row stays in L2 between its two passes (its second pass takes
  // the signs from sign words, up to V = 262144)
  const fct::FwdPlan plan = plan_forward(d, V, logits_dtype, true, true, false, nullptr, 1);
  if (fct::launch_linear(a, plan, dev, d.sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

int gemm_impl(const void* A, int64_t lda, int32_t a_mn, const void* B, int64_t ldb, int32_t b_mn,
              void* C, int64_t ldc, int32_t c_kind, int64_t M, int64_t N, int64_t K,
              void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (c_kind != FCT_GEMM_F32 && c_kind != FCT_GEMM_BF16 && c_kind != FCT_GEMM_ADD_F32)
    return FCT_ERR_UNSUPPORTED;
  if ((a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1)) return FCT_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 1) return FCT_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FCT_OK;
  // TMA coordinates and box origins are 32-bit
  if (M > fct::kGemmMaxDim || N > fct::kGemmMaxDim || K > fct::kGemmMaxDim)
    return FCT_ERR_UNSUPPORTED;
  if (!A || !B || !C) return FCT_ERR_INVALID_ARG;
  // A: M x K, B: N x K; each stored as lines of its contiguous extent
  const int64_t a_lines = a_mn ? K : M, a_cols = a_mn ? M : K;
  const int64_t b_lines = b_mn ? K : N, b_cols = b_mn ? N : K;
  const size_t ce = c_kind == FCT_GEMM_BF16 ? 2 : 4;
  if (lda < a_cols || ldb < b_cols || ldc < N) return FCT_ERR_INVALID_ARG;
  if (!span_fits(a_lines, lda, a_cols, 2) || !span_fits(b_lines, ldb, b_cols, 2) ||
      !span_fits(M, ldc, N, static_cast<int64_t>(ce)))
    return FCT_ERR_UNSUPPORTED;
  if (!fct::gemm_operand_ok(A, lda) || !fct::gemm_operand_ok(B, ldb) || !aligned(C, ce) ||
      (dev_status && !aligned(dev_status, 4)))
    return FCT_ERR_ALIGNMENT;
  const Range c = mat_range(C, M, ldc, N, ce);
  if (overlap(c, mat_range(A, a_lines, lda, a_cols, 2)) ||
      overlap(c, mat_range(B, b_lines, ldb, b_cols, 2)))
    return FCT_ERR_INVALID_ARG;
  if (workspace_bytes > 0) {
    if (workspace == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return FCT_ERR_ALIGNMENT;
    const Range w = vec_range(workspace, static_cast<int64_t>(workspace_bytes), 1);
    if (overlap(w, c) || overlap(w, mat_range(A, a_lines, lda, a_cols, 2)) ||
        overlap(w, mat_range(B, b_lines, ldb, b_cols, 2)))
      return FCT_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  const int rc = current_device(&d);
  if (rc != FCT_OK) return rc;
  if (fct::launch_gemm(fct::GemmOperand{A, lda, a_mn != 0}, fct::GemmOperand{B, ldb, b_mn != 0}, C,
                       ldc, c_kind, M, N, K, dev_status, d.sms,
                       static_cast<cudaStream_t>(stream), workspace_bytes ? workspace : nullptr,
                       workspace_bytes) != cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

// Vocabulary shards: one pass over a shard's columns (pass 1 or pass 2).
int vp_pass_impl(const void* student, int64_t ld_s, const void* teacher, int64_t ld_t, int dtype,
                 const int64_t* target, int64_t BT, int64_t V_shard, int64_t v_begin,
                 int64_t ignore_index, const float* lse_s, const float* lse_t, float* part,
                 bool tvd_pass, void* stream) {
  if (BT < 0 || v_begin < 0) return FCT_ERR_INVALID_ARG;
  if (BT == 0) return FCT_OK;
  int rc = check_common(dtype, target, BT, V_shard);
  if (rc != FCT_OK) return rc;
  if ((rc = check_logits(student, ld_s, dtype, V_shard, BT)) != FCT_OK) return rc;
  if ((rc = check_logits(teacher, ld_t, dtype, V_shard, BT)) != FCT_OK) return rc;
  if (part == nullptr) return FCT_ERR_INVALID_ARG;
  if (!aligned(part, 4)) return FCT_ERR_ALIGNMENT;
  if (tvd_pass) {
    if (lse_s == nullptr || lse_t == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(lse_s, 4) || !aligned(lse_t, 4)) return FCT_ERR_ALIGNMENT;
  }
  const size_t e = elem_size(dtype);
  const Range out = vec_range(part, BT * (tvd_pass ? 2 : 3), 4);
  if (overlap(out, mat_range(student, BT, ld_s, V_shard, e)) ||
      overlap(out, mat_range(teacher, BT, ld_t, V_shard, e)) ||
      overlap(out, vec_range(target, BT, 8)) ||
      (tvd_pass && (overlap(out, vec_range(lse_s, BT, 4)) || overlap(out, vec_range(lse_t, BT, 4)))))
    return FCT_ERR_INVALID_ARG;
  DeviceInfo d;
  if ((rc = current_device(&d)) != FCT_OK) return rc;
  fct::VpArgs a{student, teacher, ld_s, ld_t, dtype, target, BT, V_shard, v_begin, ignore_index,
                lse_s, lse_t, part};
  const bool vec = vec_ok(student, ld_s, dtype) && vec_ok(teacher, ld_t, dtype);
  if (fct::launch_vp_pass(a, vec, tvd_pass, d.sms, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

int vp_merge_impl(const float* parts, int64_t n_shards, const int64_t* target, int64_t BT,
                  int64_t V, int64_t ignore_index, float* ce, float* lse_s, float* lse_t,
                  float* tvd, float* sigma, int32_t* dev_status, bool tvd_merge, void* stream) {
  if (BT < 0 || n_shards < 1) return FCT_ERR_INVALID_ARG;
  if (BT == 0) return FCT_OK;
  if (!tvd_merge && V <= 0) return FCT_ERR_INVALID_ARG;
  if (n_shards > (int64_t(1) << 20) || BT > (int64_t(1) << 40)) return FCT_ERR_UNSUPPORTED;
  if (parts == nullptr || target == nullptr) return FCT_ERR_INVALID_ARG;
  if (!aligned(parts, 4) || !aligned(target, 8) || (dev_status && !aligned(dev_status, 4)))
    return FCT_ERR_ALIGNMENT;
  float* outs[3] = {ce, lse_s, lse_t};
  if (tvd_merge) {
    outs[0] = tvd;
    outs[1] = sigma;
    outs[2] = nullptr;
  }
  const int n_out = tvd_merge ? 2 : 3;
  const Range rp = vec_range(parts, n_shards * BT * (tvd_merge ? 2 : 3), 4);
  const Range rt = vec_range(target, BT, 8);
  for (int i = 0; i < n_out; ++i) {
    if (outs[i] == nullptr) return FCT_ERR_INVALID_ARG;
    if (!aligned(outs[i], 4)) return FCT_ERR_ALIGNMENT;
    const Range r = vec_range(outs[i], BT, 4);
    if (overlap(r, rp) || overlap(r, rt)) return FCT_ERR_INVALID_ARG;
    for (int j = i + 1; j < n_out; ++j)
      if (overlap(r, vec_range(outs[j], BT, 4))) return FCT_ERR_INVALID_ARG;
  }
  DeviceInfo d;
  const int rc = current_device(&d);
  if (rc != FCT_OK) return rc;
  fct::VpMergeArgs a{parts, n_shards, target, BT, V, ignore_index, ce, lse_s, lse_t,
                     tvd, sigma, dev_status};
  if (fct::launch_vp_merge(a, tvd_merge, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCT_ERR_CUDA;
  return FCT_OK;
}

}  // namespace

namespace fct {

int plan_linear_forward(int64_t V, int logits_dtype, FwdPlan* plan, int* device, int* sms) {
  DeviceInfo d;
  const int rc = current_device(&d);
  if (rc != FCT_OK) return rc;
  if (cudaGetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return FCT_ERR_CUDA;
  }
  *plan = plan_forward(d, V, logits_dtype, true, true);
  *sms = d.sms;
  return FCT_OK;
}

}  // namespace fct

extern "C" {

size_t fused_linear_ce_tvd_workspace_size(int64_t V, int64_t chunk_rows,
                                          fct_dtype logits_dtype) {
  if (V <= 0 || chunk_rows <= 0) return 0;
  if (logits_dtype != FCT_F32 && logits_dtype != FCT_BF16) return 0;
  const size_t b = fct::linear_workspace_bytes(V, chunk_rows, logits_dtype);
  return b == SIZE_MAX ? 0 : b;
}

int fused_linear_ce_tvd_forward_backward(
    const void* h_student, int64_t ld_h_student, const void* w_student, int64_t ld_w_student,
    int64_t d_student, const void* h_teacher, int64_t ld_h_teacher, const void* w_teacher,
    int64_t ld_w_teacher, int64_t d_teacher, const int64_t* target, int64_t BT, int64_t V,
    int64_t ignore_index, const float* grad_ce, const float* grad_tvd, int64_t grad_stride,
    float* ce, float* tvd, float* student_lse, float* teacher_lse, float* sigma,
    void* grad_h_student, int64_t ld_grad_h, float* grad_w_student, int64_t ld_grad_w,
    fct_dtype logits_dtype, void* workspace, size_t workspace_bytes, int64_t chunk_rows,
    int32_t* dev_status, void* stream) {
  return linear_impl(h_student, ld_h_student, w_student, ld_w_student, d_student, h_teacher,
                     ld_h_teacher, w_teacher, ld_w_teacher, d_teacher, target, BT, V,
                     ignore_index, grad_ce, grad_tvd, grad_stride, ce, tvd, student_lse,
                     teacher_lse, sigma, grad_h_student, ld_grad_h, grad_w_student, ld_grad_w,
                     logits_dtype, workspace, workspace_bytes, chunk_rows, dev_status, stream);
}

int fused_ce_tvd_forward_backward(const void* student, int64_t ld_student, const void* teacher,
                                  int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                                  int64_t BT, int64_t V, int64_t ignore_index,
                                  const float* grad_ce, const float* grad_tvd,
                                  int64_t grad_stride, float* ce, float* tvd,
                                  float* student_lse, float* teacher_lse, float* sigma,
                                  void* grad_student, int64_t ld_grad, int32_t* dev_status,
                                  void* stream) {
  return forward_backward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                               ignore_index, grad_ce, grad_tvd, grad_stride, ce, tvd,
                               student_lse, teacher_lse, sigma, grad_student, ld_grad,
                               dev_status, stream);
}

int fused_ce_tvd_forward_backward_ex(const void* student, int64_t ld_student,
                                     const void* teacher, int64_t ld_teacher, fct_dtype dtype,
                                     const int64_t* target, int64_t BT, int64_t V,
                                     int64_t ignore_index, const float* grad_ce,
                                     const float* grad_tvd, int64_t grad_stride, float* ce,
                                     float* tvd, float* student_lse, float* teacher_lse,
                                     float* sigma, void* grad_student, int64_t ld_grad,
                                     const fct_options* options, int32_t* dev_status,
                                     void* stream) {
  return forward_backward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                               ignore_index, grad_ce, grad_tvd, grad_stride, ce, tvd,
                               student_lse, teacher_lse, sigma, grad_student, ld_grad,
                               dev_status, stream, options);
}


int fused_ce_tvd_forward(const void* student, int64_t ld_student, const void* teacher,
                         int64_t ld_teacher, fct_dtype dtype, const int64_t* target, int64_t BT,
                         int64_t V, int64_t ignore_index, float* ce, float* tvd,
                         float* student_lse, float* teacher_lse, float* sigma,
                         int32_t* dev_status, void* stream) {
  if (teacher == nullptr || tvd == nullptr || teacher_lse == nullptr || sigma == nullptr)
    return BT == 0 ? FCT_OK : FCT_ERR_INVALID_ARG;
  return forward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                      ignore_index, ce, tvd, student_lse, teacher_lse, sigma, dev_status, stream);
}

int fused_ce_tvd_forward_ex(const void* student, int64_t ld_student, const void* teacher,
                            int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                            int64_t BT, int64_t V, int64_t ignore_index, float* ce, float* tvd,
                            float* student_lse, float* teacher_lse, float* sigma,
                            const fct_options* options, int32_t* dev_status, void* stream) {
  if (teacher == nullptr || tvd == nullptr || teacher_lse == nullptr || sigma == nullptr)
    return BT == 0 ? check_options(options) : FCT_ERR_INVALID_ARG;
  return forward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                      ignore_index, ce, tvd, student_lse, teacher_lse, sigma, dev_status, stream,
                      nullptr, 0, options);
}

int fused_ce_tvd_backward(const void* student, int64_t ld_student, const void* teacher,
                          int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                          int64_t BT, int64_t V, int64_t ignore_index, const float* student_lse,
                          const float* teacher_lse, const float* sigma, const float* grad_ce,
                          const float* grad_tvd, int64_t grad_stride, void* grad_student,
                          int64_t ld_grad, int32_t* dev_status, void* stream) {
  if (teacher == nullptr || teacher_lse == nullptr || sigma == nullptr || grad_tvd == nullptr)
    return BT == 0 ? FCT_OK : FCT_ERR_INVALID_ARG;
  return backward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                       ignore_index, student_lse, teacher_lse, sigma, grad_ce, grad_tvd,
                       grad_stride, grad_student, ld_grad, dev_status, stream);
}

int64_t fused_ce_tvd_signs_row_bytes(int64_t V, fct_dtype dtype) {
  if (V <= 0 || (dtype != FCT_F32 && dtype != FCT_BF16)) return 0;
  return signs_row_bytes(V, dtype);
}

int fused_ce_tvd_forward_signs(const void* student, int64_t ld_student, const void* teacher,
                               int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                               int64_t BT, int64_t V, int64_t ignore_index, float* ce, float* tvd,
                               float* student_lse, float* teacher_lse, float* sigma,
                               uint8_t* signs, int64_t ld_signs, int32_t* dev_status,
                               void* stream) {
  if (teacher == nullptr || tvd == nullptr || teacher_lse == nullptr || sigma == nullptr ||
      signs == nullptr)
    return BT == 0 ? FCT_OK : FCT_ERR_INVALID_ARG;
  return forward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                      ignore_index, ce, tvd, student_lse, teacher_lse, sigma, dev_status, stream,
                      signs, ld_signs);
}

int fused_ce_tvd_forward_signs_ex(const void* student, int64_t ld_student, const void* teacher,
                                  int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                                  int64_t BT, int64_t V, int64_t ignore_index, float* ce,
                                  float* tvd, float* student_lse, float* teacher_lse,
                                  float* sigma, uint8_t* signs, int64_t ld_signs,
                                  const fct_options* options, int32_t* dev_status,
                                  void* stream) {
  if (teacher == nullptr || tvd == nullptr || teacher_lse == nullptr || sigma == nullptr ||
      signs == nullptr)
    return BT == 0 ? check_options(options) : FCT_ERR_INVALID_ARG;
  return forward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                      ignore_index, ce, tvd, student_lse, teacher_lse, sigma, dev_status, stream,
                      signs, ld_signs, options);
}

int fused_ce_tvd_backward_signs(const void* student, int64_t ld_student, const void* teacher,
                                int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                                int64_t BT, int64_t V, int64_t ignore_index,
                                const float* student_lse, const float* teacher_lse,
                                const float* sigma, const uint8_t* signs, int64_t ld_signs,
                                const float* grad_ce, const float* grad_tvd, int64_t grad_stride,
                                void* grad_student, int64_t ld_grad, int32_t* dev_status,
                                void* stream) {
  if (teacher == nullptr || teacher_lse == nullptr || sigma == nullptr || grad_tvd == nullptr ||
      signs == nullptr)
    return BT == 0 ? FCT_OK : FCT_ERR_INVALID_ARG;
  return backward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V,
                       ignore_index, student_lse, teacher_lse, sigma, grad_ce, grad_tvd,
                       grad_stride, grad_student, ld_grad, dev_status, stream, signs, ld_signs);
}

int ce_forward_backward(const void* logits, int64_t ld, fct_dtype dtype, const int64_t* target,
                        int64_t BT, int64_t V, int64_t ignore_index, const float* grad_ce,
                        int64_t grad_stride, float* ce, float* lse, void* grad_logits,
                        int64_t ld_grad, int32_t* dev_status, void* stream) {
  return ce_forward_backward_impl(logits, ld, dtype, target, BT, V, ignore_index, grad_ce,
                                  grad_stride, ce, lse, grad_logits, ld_grad, dev_status, stream);
}

int ce_forward_backward_ex(const void* logits, int64_t ld, fct_dtype dtype,
                           const int64_t* target, int64_t BT, int64_t V, int64_t ignore_index,
                           const float* grad_ce, int64_t grad_stride, float* ce, float* lse,
                           void* grad_logits, int64_t ld_grad, const fct_options* options,
                           int32_t* dev_status, void* stream) {
  return ce_forward_backward_impl(logits, ld, dtype, target, BT, V, ignore_index, grad_ce,
                                  grad_stride, ce, lse, grad_logits, ld_grad, dev_status, stream,
                                  options);
}

int ce_forward(const void* logits, int64_t ld, fct_dtype dtype, const int64_t* target, int64_t BT,
               int64_t V, int64_t ignore_index, float* ce, float* lse, int32_t* dev_status,
               void* stream) {
  return forward_impl(logits, ld, nullptr, ld, dtype, target, BT, V, ignore_index, ce, nullptr,
                      lse, nullptr, nullptr, dev_status, stream);
}

int ce_forward_ex(const void* logits, int64_t ld, fct_dtype dtype, const int64_t* target,
                  int64_t BT, int64_t V, int64_t ignore_index, float* ce, float* lse,
                  const fct_options* options, int32_t* dev_status, void* stream) {
  return forward_impl(logits, ld, nullptr, ld, dtype, target, BT, V, ignore_index, ce, nullptr,
                      lse, nullptr, nullptr, dev_status, stream, nullptr, 0, options);
}

int ce_backward(const void* logits, int64_t ld, fct_dtype dtype, const int64_t* target,
                int64_t BT, int64_t V, int64_t ignore_index, const float* lse,
                const float* grad_ce, int64_t grad_stride, void* grad_logits, int64_t ld_grad,
                int32_t* dev_status, void* stream) {
  return backward_impl(logits, ld, nullptr, ld, dtype, target, BT, V, ignore_index, lse, nullptr,
                       nullptr, grad_ce, nullptr, grad_stride, grad_logits, ld_grad, dev_status,
                       stream);
}

int fused_ce_tvd_mean_upstream(const int64_t* target, int64_t BT, int64_t ignore_index,
                               double alpha, double beta, float* grad_ce, float* grad_tvd,
                               int64_t* count, void* stream) {
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  if (target == nullptr || grad_ce == nullptr || grad_tvd == nullptr) return FCT_ERR_INVALID_ARG;
  if (!aligned(target, 8) || !aligned(grad_ce, 4) || !aligned(grad_tvd, 4) ||
      (count && !aligned(count, 8)))
    return FCT_ERR_ALIGNMENT;
  if (grad_ce == grad_tvd) return FCT_ERR_INVALID_ARG;
  DeviceInfo d;
  const int rc = current_device(&d);
  if (rc != FCT_OK) return rc;
  fct::LossArgs a{target, BT, ignore_index, nullptr, nullptr, alpha, beta,
                  nullptr, grad_ce, grad_tvd, count};
  return fct::launch_mean(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FCT_OK
                                                                                : FCT_ERR_CUDA;
}

int fused_ce_tvd_mean_loss(const float* ce, const float* tvd, const int64_t* target, int64_t BT,
                           int64_t ignore_index, double alpha, double beta, float* loss,
                           void* stream) {
  if (BT < 0) return FCT_ERR_INVALID_ARG;
  if (ce == nullptr || tvd == nullptr || target == nullptr || loss == nullptr)
    return FCT_ERR_INVALID_ARG;
  if (!aligned(ce, 4) || !aligned(tvd, 4) || !aligned(target, 8) || !aligned(loss, 4))
    return FCT_ERR_ALIGNMENT;
  const Range l = vec_range(loss, 1, 4);
  if (overlap(l, vec_range(ce, BT, 4)) || overlap(l, vec_range(tvd, BT, 4)) ||
      overlap(l, vec_range(target, BT, 8)))
    return FCT_ERR_INVALID_ARG;
  DeviceInfo d;
  const int rc = current_device(&d);
  if (rc != FCT_OK) return rc;
  fct::LossArgs a{target, BT, ignore_index, ce, tvd, alpha, beta,
                  loss, nullptr, nullptr, nullptr};
  return fct::launch_mean(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FCT_OK
                                                                                : FCT_ERR_CUDA;
}

int fused_ce_tvd_vp_lse(const void* student, int64_t ld_student, const void* teacher,
                        int64_t ld_teacher, fct_dtype dtype, const int64_t* target, int64_t BT,
                        int64_t V_shard, int64_t v_begin, int64_t ignore_index, float* part,
                        void* stream) {
  return vp_pass_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V_shard,
                      v_begin, ignore_index, nullptr, nullptr, part, false, stream);
}

int fused_ce_tvd_vp_merge_lse(const float* parts, int64_t n_shards, const int64_t* target,
                              int64_t BT, int64_t V, int64_t ignore_index, float* ce,
                              float* student_lse, float* teacher_lse, int32_t* dev_status,
                              void* stream) {
  return vp_merge_impl(parts, n_shards, target, BT, V, ignore_index, ce, student_lse,
                       teacher_lse, nullptr, nullptr, dev_status, false, stream);
}

int fused_ce_tvd_vp_tvd(const void* student, int64_t ld_student, const void* teacher,
                        int64_t ld_teacher, fct_dtype dtype, const int64_t* target, int64_t BT,
                        int64_t V_shard, int64_t ignore_index, const float* student_lse,
                        const float* teacher_lse, float* part, void* stream) {
  return vp_pass_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V_shard, 0,
                      ignore_index, student_lse, teacher_lse, part, true, stream);
}

int fused_ce_tvd_vp_merge_tvd(const float* parts, int64_t n_shards, const int64_t* target,
                              int64_t BT, int64_t ignore_index, float* tvd, float* sigma,
                              void* stream) {
  return vp_merge_impl(parts, n_shards, target, BT, 1, ignore_index, nullptr, nullptr, nullptr,
                       tvd, sigma, nullptr, true, stream);
}

int fused_ce_tvd_vp_backward(const void* student, int64_t ld_student, const void* teacher,
                             int64_t ld_teacher, fct_dtype dtype, const int64_t* target,
                             int64_t BT, int64_t V_shard, int64_t v_begin, int64_t V,
                             int64_t ignore_index, const float* student_lse,
                             const float* teacher_lse, const float* sigma, const float* grad_ce,
                             const float* grad_tvd, int64_t grad_stride, void* grad_student,
                             int64_t ld_grad, int32_t* dev_status, void* stream) {
  if (v_begin < 0 || V_shard <= 0 || V < V_shard || v_begin > V - V_shard)
    return BT == 0 ? FCT_OK : FCT_ERR_INVALID_ARG;
  if (teacher == nullptr || teacher_lse == nullptr || sigma == nullptr || grad_tvd == nullptr)
    return BT == 0 ? FCT_OK : FCT_ERR_INVALID_ARG;
  return backward_impl(student, ld_student, teacher, ld_teacher, dtype, target, BT, V_shard,
                       ignore_index, student_lse, teacher_lse, sigma, grad_ce, grad_tvd,
                       grad_stride, grad_student, ld_grad, dev_status, stream, nullptr, 0,
                       v_begin, V);
}

const char* fct_status_string(int status) {
  switch (status) {
    case FCT_OK: return "FCT_OK";
    case FCT_ERR_INVALID_ARG: return "FCT_ERR_INVALID_ARG: invalid argument";
    case FCT_ERR_UNSUPPORTED: return "FCT_ERR_UNSUPPORTED: unsupported dtype or device";
    case FCT_ERR_ALIGNMENT: return "FCT_ERR_ALIGNMENT: pointer not aligned to its element size";
    case FCT_ERR_CUDA: return "FCT_ERR_CUDA: CUDA runtime or launch error";
    default: return "unknown fct_status";
  }
}

int fct_gemm_bf16(const void* A, int64_t lda, int32_t a_mn_major, const void* B, int64_t ldb,
                  int32_t b_mn_major, void* C, int64_t ldc, int32_t c_kind, int64_t M, int64_t N,
                  int64_t K, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                  void* stream) {
  return gemm_impl(A, lda, a_mn_major, B, ldb, b_mn_major, C, ldc, c_kind, M, N, K, workspace,
                   workspace_bytes, dev_status, stream);
}

size_t fct_gemm_bf16_workspace_size(int64_t M, int64_t N) {
  if (M <= 0 || N <= 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return 0;
  return fct::gemm_split_workspace_bytes(M, N);
}

int fct_version(void) { return 500; }  // 0.5.0: tensor-core GEMM entry point, lse partials in the fused-linear workspace

}  // extern "C"
