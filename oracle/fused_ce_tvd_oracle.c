/*
 * Fused cross-entropy + total-variation-distance loss: CPU fp64 ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Source of the method ("PR #1384 analysis" below): the blog post
 * "[Liger-Kernel] Liger-Kernel: Cross-Entropy와 Total Variation Distance를
 * 하나로 융합하여 성능을 극대화하다", an analysis of linkedin/Liger-Kernel
 * PR #1384 (fused CE + TV distance kernel).  Sections used:
 *   - "Forward Pass", step 1: per-row log-sum-exp of student and teacher;
 *   - "Forward Pass", step 2: p, q from those lse values, TVD = 0.5*sum|p-q|
 *     and sigma = sum_v p_v * sign(p_v - q_v); ce = student_lse - student[target];
 *   - "Backward Pass": d ce / d s_v = p_v - 1[v == target] and
 *     d tvd / d s_v = 0.5 * p_v * (sign_v - sigma); ignore_index rows and a
 *     zero subgradient at ties (p_v == q_v).
 * The Liger-Kernel overview page ("기술 구현") states the kernels compute
 * exactly, without approximation, so the oracle is the plain definition:
 * two-pass (exact max, then sum of exponentials, then log) in fp64, one row
 * at a time, no blocking or fusion.
 *
 * Readings where the pages are silent:
 *   - ignore rows: ce = tvd = lse_s = lse_t = sigma = 0 and a zero gradient row;
 *   - target outside [0, V) and not ignore_index: the row's ce is NaN, its
 *     gradient row is NaN, other outputs are computed, and bit 0x1 is set
 *     in the returned status;
 *   - sign(0) = 0: a tie contributes nothing to sigma and takes a zero
 *     subgradient.
 *
 * Element types of the logit matrices: 0 = fp32, 1 = bf16 (raw 16-bit
 * patterns, upcast exactly), 2 = fp64.  Rows are `ld` elements apart.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2
#define ORACLE_TARGET_OUT_OF_RANGE 0x1

/* Exact widening of one stored element to double. */
static double elem(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F32) {
    float f;
    memcpy(&f, (const char*)base + idx * 4, 4);
    return (double)f;
  }
  if (dtype == ORACLE_BF16) {
    uint16_t h;
    memcpy(&h, (const char*)base + idx * 2, 2);
    uint32_t bits = ((uint32_t)h) << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
  double d;
  memcpy(&d, (const char*)base + idx * 8, 8);
  return d;
}

/* "Forward Pass" step 1: lse = max + log(sum exp(x - max)), taken as two
 * exact passes over the row (the max first, then the sum). */
static double row_lse(const void* x, int dtype, int64_t off, int64_t V) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double xv = elem(x, dtype, off + v);
    if (xv > m) m = xv;
  }
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) s += exp(elem(x, dtype, off + v) - m);
  return m + log(s);
}

static double sgn(double d) { return (d > 0.0) - (d < 0.0); }

/* Softmax probabilities of one student row (p) and one teacher row (q). */
void oracle_row_probs(const void* student, int64_t ld_s, const void* teacher,
                      int64_t ld_t, int dtype, int64_t row, int64_t V,
                      double* p, double* q) {
  int64_t os = row * ld_s, ot = row * ld_t;
  double lse_s = row_lse(student, dtype, os, V);
  double lse_t = row_lse(teacher, dtype, ot, V);
  for (int64_t v = 0; v < V; ++v) {
    p[v] = exp(elem(student, dtype, os + v) - lse_s);
    q[v] = exp(elem(teacher, dtype, ot + v) - lse_t);
  }
}

/* Forward: per row ce, tvd, student_lse, teacher_lse, sigma ("Forward Pass",
 * steps 1 and 2 and the per-row stores that close it). */
int oracle_fused_ce_tvd_forward(const void* student, int64_t ld_s,
                                const void* teacher, int64_t ld_t, int dtype,
                                const int64_t* target, int64_t BT, int64_t V,
                                int64_t ignore_index, double* ce, double* tvd,
                                double* lse_s_out, double* lse_t_out,
                                double* sigma_out, int nthreads) {
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : status)
  for (int64_t r = 0; r < BT; ++r) {
    int64_t tg = target[r];
    if (tg == ignore_index) {
      ce[r] = tvd[r] = lse_s_out[r] = lse_t_out[r] = sigma_out[r] = 0.0;
      continue;
    }
    int64_t os = r * ld_s, ot = r * ld_t;
    double lse_s = row_lse(student, dtype, os, V);
    double lse_t = row_lse(teacher, dtype, ot, V);
    double abs_sum = 0.0, sigma = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      double p = exp(elem(student, dtype, os + v) - lse_s);
      double q = exp(elem(teacher, dtype, ot + v) - lse_t);
      double d = p - q;
      abs_sum += fabs(d);
      sigma += p * sgn(d);
    }
    if (tg < 0 || tg >= V) {
      status |= ORACLE_TARGET_OUT_OF_RANGE;
      ce[r] = NAN;
    } else {
      ce[r] = lse_s - elem(student, dtype, os + tg);
    }
    tvd[r] = 0.5 * abs_sum;
    lse_s_out[r] = lse_s;
    lse_t_out[r] = lse_t;
    sigma_out[r] = sigma;
  }
  return status;
}

/* Backward ("Backward Pass"): recomputes every quantity of the row from the
 * logits and writes
 *   g_v = grad_ce * (p_v - 1[v == target]) + grad_tvd * 0.5 * p_v * (sign_v - sigma)
 * into grad (fp64, BT x V, dense).  grad_stride = 1 reads one upstream value
 * per row, 0 broadcasts element 0. */
int oracle_fused_ce_tvd_backward(const void* student, int64_t ld_s,
                                 const void* teacher, int64_t ld_t, int dtype,
                                 const int64_t* target, int64_t BT, int64_t V,
                                 int64_t ignore_index, const double* grad_ce,
                                 const double* grad_tvd, int64_t grad_stride,
                                 double* grad, int nthreads) {
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : status)
  for (int64_t r = 0; r < BT; ++r) {
    double* g = grad + r * V;
    int64_t tg = target[r];
    if (tg == ignore_index) {
      for (int64_t v = 0; v < V; ++v) g[v] = 0.0;
      continue;
    }
    if (tg < 0 || tg >= V) {
      status |= ORACLE_TARGET_OUT_OF_RANGE;
      for (int64_t v = 0; v < V; ++v) g[v] = NAN;
      continue;
    }
    int64_t os = r * ld_s, ot = r * ld_t;
    double lse_s = row_lse(student, dtype, os, V);
    double lse_t = row_lse(teacher, dtype, ot, V);
    double sigma = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      double p = exp(elem(student, dtype, os + v) - lse_s);
      double q = exp(elem(teacher, dtype, ot + v) - lse_t);
      sigma += p * sgn(p - q);
    }
    double gce = grad_ce[r * grad_stride], gtvd = grad_tvd[r * grad_stride];
    for (int64_t v = 0; v < V; ++v) {
      double p = exp(elem(student, dtype, os + v) - lse_s);
      double q = exp(elem(teacher, dtype, ot + v) - lse_t);
      double onehot = (v == tg) ? 1.0 : 0.0;
      g[v] = gce * (p - onehot) + gtvd * 0.5 * p * (sgn(p - q) - sigma);
    }
  }
  return status;
}

/* Cross-entropy alone: ce = lse - x[target] (the CE half of "Forward Pass"). */
int oracle_ce_forward(const void* logits, int64_t ld, int dtype,
                      const int64_t* target, int64_t BT, int64_t V,
                      int64_t ignore_index, double* ce, double* lse_out,
                      int nthreads) {
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : status)
  for (int64_t r = 0; r < BT; ++r) {
    int64_t tg = target[r];
    if (tg == ignore_index) {
      ce[r] = lse_out[r] = 0.0;
      continue;
    }
    double lse = row_lse(logits, dtype, r * ld, V);
    lse_out[r] = lse;
    if (tg < 0 || tg >= V) {
      status |= ORACLE_TARGET_OUT_OF_RANGE;
      ce[r] = NAN;
    } else {
      ce[r] = lse - elem(logits, dtype, r * ld + tg);
    }
  }
  return status;
}

/* Cross-entropy gradient alone: g_v = grad_ce * (p_v - 1[v == target])
 * (the first line of the "Backward Pass" identities). */
int oracle_ce_backward(const void* logits, int64_t ld, int dtype,
                       const int64_t* target, int64_t BT, int64_t V,
                       int64_t ignore_index, const double* grad_ce,
                       int64_t grad_stride, double* grad, int nthreads) {
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : status)
  for (int64_t r = 0; r < BT; ++r) {
    double* g = grad + r * V;
    int64_t tg = target[r];
    if (tg == ignore_index) {
      for (int64_t v = 0; v < V; ++v) g[v] = 0.0;
      continue;
    }
    if (tg < 0 || tg >= V) {
      status |= ORACLE_TARGET_OUT_OF_RANGE;
      for (int64_t v = 0; v < V; ++v) g[v] = NAN;
      continue;
    }
    double lse = row_lse(logits, dtype, r * ld, V);
    double gce = grad_ce[r * grad_stride];
    for (int64_t v = 0; v < V; ++v) {
      double p = exp(elem(logits, dtype, r * ld + v) - lse);
      g[v] = gce * (p - ((v == tg) ? 1.0 : 0.0));
    }
  }
  return status;
}

/* Mean over tokens (the caller-side reduction the method leaves open):
 * loss = (alpha * sum_r ce_r + beta * sum_r tvd_r) / n over the n rows whose
 * target is not ignore_index; *grad_ce = alpha / n and *grad_tvd = beta / n
 * are its derivatives with respect to each kept row's ce and tvd (all 0 when
 * n = 0).  Returns n. */
int64_t oracle_mean_loss(const double* ce, const double* tvd, const int64_t* target,
                         int64_t BT, int64_t ignore_index, double alpha, double beta,
                         double* loss, double* grad_ce, double* grad_tvd) {
  int64_t n = 0;
  double sce = 0.0, stvd = 0.0;
  for (int64_t r = 0; r < BT; ++r) {
    if (target[r] == ignore_index) continue;
    n += 1;
    sce += ce[r];
    stvd += tvd[r];
  }
  *loss = n ? (alpha * sce + beta * stvd) / (double)n : 0.0;
  *grad_ce = n ? alpha / (double)n : 0.0;
  *grad_tvd = n ? beta / (double)n : 0.0;
  return n;
}
