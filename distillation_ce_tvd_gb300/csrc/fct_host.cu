// Single-launch forward + backward from and to host memory.
//
// The loss's inputs often live in host memory (a data loader's pinned
// buffers, logits streamed from another device).  This entry point moves row
// blocks through a ring of device slots in the caller's workspace with three
// streams: block i is copied in on a copy-in stream while block i-1 is
// computed on the caller's stream and block i-2's gradient and per-row
// outputs are copied back on a copy-out stream.  Every copy is one
// cudaMemcpyAsync (or cudaMemcpy2DAsync for padded rows); events order the
// three streams.  Each
// block's gradient is computed in place over its student slot (the
// single-launch kernel's in-place mode) and copied out from there, so a slot
// holds two logit blocks and a few per-row vectors.  Rows are independent,
// so the results equal one device call on the whole batch, bit for bit.
#include "fct_internal.h"

namespace {

constexpr int kSlots = 3;          // ring of device slots: in, compute, out
constexpr size_t kAlign = 256;     // every workspace region starts on 256 bytes

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t elem_bytes(int dtype) { return dtype == FCT_BF16 ? 2 : 4; }

// Device row stride of a slot's logit blocks: a multiple of 16 bytes, so the
// kernel's 16-byte vector path always applies.
int64_t slot_ld(int64_t V, int dtype) {
  const int64_t vec = 16 / static_cast<int64_t>(elem_bytes(dtype));
  return (V + vec - 1) / vec * vec;
}

struct SlotLayout {
  size_t logits;   // bytes of one (rows, slot_ld) logit block
  size_t target;   // rows int64
  size_t rowvec;   // rows fp32
  size_t slot;     // whole slot
};

SlotLayout layout(int64_t V, int dtype, int64_t rows) {
  SlotLayout L;
  L.logits = round_up(size_t(rows) * size_t(slot_ld(V, dtype)) * elem_bytes(dtype), kAlign);
  L.target = round_up(size_t(rows) * 8, kAlign);
  L.rowvec = round_up(size_t(rows) * 4, kAlign);
  // student (and gradient), teacher, target, grad_ce, grad_tvd, 5 outputs
  L.slot = 2 * L.logits + L.target + 7 * L.rowvec;
  return L;
}

// Largest V and block_rows for which every size above fits comfortably in
// 64 bits (a 2^62-byte workspace is far beyond any device).
bool sizes_ok(int64_t V, int64_t rows) {
  return V > 0 && rows > 0 && V <= (int64_t(1) << 40) && rows <= (int64_t(1) << 20);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// One copy of `rows` rows of `width` bytes: a plain copy when both sides are
// contiguous (the copy engines then move one linear range), else a pitched
// copy.
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t st) {
  if (dpitch == width && spitch == width) return cudaMemcpyAsync(dst, src, width * rows, kind, st);
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st);
}

// Streams and events of one call, released when the call returns (the
// runtime defers the release until their work is done).
struct Pipeline {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t copied[kSlots] = {}, computed[kSlots] = {}, returned[kSlots] = {};

  cudaError_t create() {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t* all[] = {&start, &end};
    for (cudaEvent_t* ev : all)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int j = 0; j < kSlots; ++j) {
      if ((e = cudaEventCreateWithFlags(&copied[j], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&computed[j], cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&returned[j], cudaEventDisableTiming)) != cudaSuccess)
        return e;
    }
    return cudaSuccess;
  }

  ~Pipeline() {
    for (int j = 0; j < kSlots; ++j) {
      if (copied[j]) cudaEventDestroy(copied[j]);
      if (computed[j]) cudaEventDestroy(computed[j]);
      if (returned[j]) cudaEventDestroy(returned[j]);
    }
    if (start) cudaEventDestroy(start);
    if (end) cudaEventDestroy(end);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
};

}  // namespace

extern "C" {

size_t fused_ce_tvd_host_workspace_size(int64_t V, fct_dtype dtype, int64_t block_rows) {
  if (dtype != FCT_F32 && dtype != FCT_BF16) return 0;
  if (!sizes_ok(V, block_rows)) return 0;
  return kAlign + kSlots * layout(V, dtype, block_rows).slot;
}

int fused_ce_tvd_forward_backward_host(
    const void* student, int64_t ld_student, const void* teacher, int64_t ld_teacher,
    fct_dtype dtype, const int64_t* target, int64_t BT, int64_t V, int64_t ignore_index,
    const float* grad_ce, const float* grad_tvd, int64_t grad_stride, float* ce, float* tvd,
    float* student_lse, float* teacher_lse, float* sigma, void* grad_student, int64_t ld_grad,
    void* workspace, size_t workspace_bytes, int64_t block_rows, int32_t* status,
    void* stream) {
  if (BT < 0 || block_rows <= 0) return FCT_ERR_INVALID_ARG;
  if (dtype != FCT_F32 && dtype != FCT_BF16) return FCT_ERR_UNSUPPORTED;
  if (BT == 0) return FCT_OK;
  if (!sizes_ok(V, block_rows)) return V <= 0 ? FCT_ERR_INVALID_ARG : FCT_ERR_UNSUPPORTED;
  if (!student || !teacher || !target || !grad_ce || !grad_tvd || !workspace)
    return FCT_ERR_INVALID_ARG;
  if (ld_student < V || ld_teacher < V || (grad_student && ld_grad < V))
    return FCT_ERR_INVALID_ARG;
  if (grad_stride != 0 && grad_stride != 1) return FCT_ERR_INVALID_ARG;
  const size_t e = elem_bytes(dtype);
  if (!aligned(student, e) || !aligned(teacher, e) || (grad_student && !aligned(grad_student, e)) ||
      !aligned(target, 8) || !aligned(grad_ce, 4) || !aligned(grad_tvd, 4) ||
      !aligned(workspace, kAlign) || (status && !aligned(status, 4)))
    return FCT_ERR_ALIGNMENT;
  float* outs[5] = {ce, tvd, student_lse, teacher_lse, sigma};
  for (float* o : outs)
    if (o && !aligned(o, 4)) return FCT_ERR_ALIGNMENT;
  const int64_t rows = block_rows < BT ? block_rows : BT;
  const SlotLayout L = layout(V, dtype, rows);
  if (workspace_bytes < kAlign + kSlots * L.slot) return FCT_ERR_INVALID_ARG;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Pipeline P;
  if (P.create() != cudaSuccess) {
    cudaGetLastError();
    return FCT_ERR_CUDA;
  }
  char* ws = static_cast<char*>(workspace);
  int32_t* dev_status = reinterpret_cast<int32_t*>(ws);
  const int64_t ldd = slot_ld(V, dtype);
  const size_t dpitch = size_t(ldd) * e, width = size_t(V) * e;
  const auto* S = static_cast<const char*>(student);
  const auto* T = static_cast<const char*>(teacher);
  auto* G = static_cast<char*>(grad_student);

  // Nothing may overwrite the workspace before the caller's earlier work on
  // `stream` is done with it.
  bool ok = cudaEventRecord(P.start, st) == cudaSuccess &&
            cudaStreamWaitEvent(P.in, P.start, 0) == cudaSuccess &&
            cudaMemsetAsync(dev_status, 0, sizeof(int32_t), P.in) == cudaSuccess;
  int rc = FCT_OK;
  int64_t i = 0;
  for (int64_t r0 = 0; ok && r0 < BT; r0 += rows, ++i) {
    const int64_t R = (BT - r0 < rows) ? BT - r0 : rows;
    const int j = static_cast<int>(i % kSlots);
    char* slot = ws + kAlign + j * L.slot;
    char* s_dev = slot;                                  // student, then its gradient
    char* t_dev = slot + L.logits;
    auto* tg_dev = reinterpret_cast<int64_t*>(slot + 2 * L.logits);
    auto* gce_dev = reinterpret_cast<float*>(slot + 2 * L.logits + L.target);
    auto* gtvd_dev = reinterpret_cast<float*>(slot + 2 * L.logits + L.target + L.rowvec);
    float* out_dev[5];
    for (int k = 0; k < 5; ++k)
      out_dev[k] = reinterpret_cast<float*>(slot + 2 * L.logits + L.target + (2 + k) * L.rowvec);
    const int64_t n_up = grad_stride ? R : 1;
    const int64_t up0 = grad_stride ? r0 : 0;

    // copy in (after the copy-out of the block that last used this slot)
    ok = (i < kSlots || cudaStreamWaitEvent(P.in, P.returned[j], 0) == cudaSuccess) &&
         copy_rows(s_dev, dpitch, S + size_t(r0) * size_t(ld_student) * e,
                   size_t(ld_student) * e, width, size_t(R), cudaMemcpyHostToDevice,
                   P.in) == cudaSuccess &&
         copy_rows(t_dev, dpitch, T + size_t(r0) * size_t(ld_teacher) * e,
                   size_t(ld_teacher) * e, width, size_t(R), cudaMemcpyHostToDevice,
                   P.in) == cudaSuccess &&
         cudaMemcpyAsync(tg_dev, target + r0, size_t(R) * 8, cudaMemcpyHostToDevice, P.in) ==
             cudaSuccess &&
         cudaMemcpyAsync(gce_dev, grad_ce + up0, size_t(n_up) * 4, cudaMemcpyHostToDevice,
                         P.in) == cudaSuccess &&
         cudaMemcpyAsync(gtvd_dev, grad_tvd + up0, size_t(n_up) * 4, cudaMemcpyHostToDevice,
                         P.in) == cudaSuccess &&
         cudaEventRecord(P.copied[j], P.in) == cudaSuccess;
    if (!ok) break;
    // compute, in place over the student slot
    if (cudaStreamWaitEvent(st, P.copied[j], 0) != cudaSuccess) {
      ok = false;
      break;
    }
    rc = fused_ce_tvd_forward_backward_ex(s_dev, ldd, t_dev, ldd, dtype, tg_dev, R, V,
                                          ignore_index, gce_dev, gtvd_dev, grad_stride,
                                          out_dev[0], out_dev[1], out_dev[2], out_dev[3],
                                          out_dev[4], s_dev, ldd, nullptr, dev_status, st);
    if (rc != FCT_OK) break;
    // copy out
    ok = cudaEventRecord(P.computed[j], st) == cudaSuccess &&
         cudaStreamWaitEvent(P.out, P.computed[j], 0) == cudaSuccess;
    if (ok && G)
      ok = copy_rows(G + size_t(r0) * size_t(ld_grad) * e, size_t(ld_grad) * e, s_dev, dpitch,
                     width, size_t(R), cudaMemcpyDeviceToHost, P.out) == cudaSuccess;
    for (int k = 0; ok && k < 5; ++k)
      if (outs[k])
        ok = cudaMemcpyAsync(outs[k] + r0, out_dev[k], size_t(R) * 4, cudaMemcpyDeviceToHost,
                             P.out) == cudaSuccess;
    ok = ok && cudaEventRecord(P.returned[j], P.out) == cudaSuccess;
  }
  if (ok && rc == FCT_OK && status)
    ok = cudaMemcpyAsync(status, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, P.out) ==
         cudaSuccess;
  // The caller's stream owns the workspace and the host buffers again once
  // everything enqueued above is done (also after a failure part-way).
  const bool joined = cudaEventRecord(P.end, P.out) == cudaSuccess &&
                      cudaStreamWaitEvent(st, P.end, 0) == cudaSuccess &&
                      cudaEventRecord(P.start, P.in) == cudaSuccess &&
                      cudaStreamWaitEvent(st, P.start, 0) == cudaSuccess;
  if (rc != FCT_OK) return rc;
  if (!ok || !joined) {
    cudaGetLastError();
    return FCT_ERR_CUDA;
  }
  return FCT_OK;
}

}  // extern "C"
