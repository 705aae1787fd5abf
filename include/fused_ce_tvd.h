/*
 * fused_ce_tvd.h -- C ABI of libfused_ce_tvd.so, the GB300 (sm_103a) fused
 * cross-entropy + total-variation-distance distillation loss.
 *
 * The method is the one described in "[Liger-Kernel] Liger-Kernel:
 * Cross-Entropy와 Total Variation Distance를 하나로 융합하여 성능을
 * 극대화하다" (an analysis of linkedin/Liger-Kernel PR #1384, "fused CE + TV
 * distance kernel"), cited below as "PR #1384 analysis".  For one row of
 * student logits s and teacher logits t over a vocabulary of V entries:
 *
 *   p = softmax(s), q = softmax(t)
 *   ce    = lse(s) - s[target]
 *   tvd   = 0.5 * sum_v |p_v - q_v|
 *   sigma = sum_v p_v * sign(p_v - q_v)            (sign(0) = 0)
 *   d(grad_ce*ce + grad_tvd*tvd)/ds_v
 *         = grad_ce*(p_v - 1[v==target]) + grad_tvd*0.5*p_v*(sign_v - sigma)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array arguments are DEVICE pointers, owned by the caller (except
 *    in the host-buffer entry point, which says which of its pointers are
 *    host memory).  The library allocates no device memory and keeps no
 *    state between calls that changes results or launches (it caches device
 *    properties, per-kernel occupancy and the driver's tensor-map encoder;
 *    the no-allocation fused-linear variant uses a fixed device array of
 *    the library).
 *  - Logit matrices are row-major (BT, V) with a row stride `ld` (in
 *    elements, ld >= V).  Student and teacher share one element type.
 *  - `target` is int64 (BT,).  A row whose target equals `ignore_index`
 *    contributes nothing: its ce, tvd, lse and sigma outputs are written as 0
 *    and its gradient row as 0.  A target outside [0, V) that is not
 *    ignore_index sets FCT_DEV_TARGET_OUT_OF_RANGE in *dev_status; that row's
 *    ce is NaN and its gradient row is NaN, the other outputs are computed.
 *  - Per-row outputs and inputs (ce, tvd, lse, sigma, grad_ce, grad_tvd) are
 *    fp32 arrays of BT values.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    are asynchronous and stream-ordered; none synchronises the host.
 *  - `dev_status` may be NULL.  Otherwise it points to one device int32 that
 *    kernels OR error bits into (never cleared by the library); read it after
 *    synchronising the stream.  No kernel traps or asserts.
 *  - The return value is a fct_status.  Argument errors are detected on the
 *    host before any launch and leave every output untouched.  A launch
 *    failure returns FCT_ERR_CUDA (the CUDA error is left for
 *    cudaGetLastError to report again).
 *  - BT == 0 is a valid no-op.  Rows are independent: splitting BT into
 *    contiguous blocks across calls (or processes) gives bitwise the same
 *    results as one call.
 */
#ifndef FUSED_CE_TVD_H_
#define FUSED_CE_TVD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FCT_F32 = 0, FCT_BF16 = 1 } fct_dtype;

typedef enum {
  FCT_OK = 0,
  FCT_ERR_INVALID_ARG = 1, /* null pointer, negative size, ld < V, bad aliasing */
  FCT_ERR_UNSUPPORTED = 2, /* unknown dtype, no sm_103a device */
  FCT_ERR_ALIGNMENT = 3,   /* pointer not aligned to its element size */
  FCT_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} fct_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define FCT_DEV_TARGET_OUT_OF_RANGE 0x1
#define FCT_DEV_WAIT_TIMEOUT 0x2 /* a bounded wait in a kernel gave up; outputs invalid */

/*
 * Launch options of the multi-pass forward kernels (a tuning and measurement
 * aid with no counterpart in the method's description).  Every entry point
 * without the _ex suffix behaves as its _ex form with options == NULL; a
 * NULL pointer and a zero-initialised struct both mean "automatic".  The
 * options belong to the one call they are passed to: the library keeps no
 * tuning state between calls.
 *
 *   ctas_per_row : 0 = automatic (depends on V, the element type and the
 *                  device only, never on BT); 1, 2, 4 or 8 = the CTAs of one
 *                  thread-block cluster that share a row.  The per-row
 *                  reduction order follows it, so results can differ in the
 *                  last bits between settings; a forward and the backward or
 *                  single launch it is compared with should use the same.
 *                  Anything else: FCT_ERR_INVALID_ARG.
 *   l2_keep      : 0 = rows that a later pass reads again are tagged
 *                  evict_last in L2; 1 = evict_normal.  Anything else:
 *                  FCT_ERR_INVALID_ARG.
 *   stagger      : start stagger of the multi-pass kernels, as a fraction of
 *                  an estimated row time: 0 = automatic (0.5), > 0 = that
 *                  fraction (at most 4), < 0 = none.  Results do not depend
 *                  on it.
 *   ring         : how the fused forward kernels (alone, with sign words,
 *                  or with the backward) stage logits in shared memory:
 *                  2 = one producer warp fills a CTA-wide ring with TMA bulk
 *                  copies (cp.async.bulk, mbarrier completion), available
 *                  where a row belongs to one CTA; 1 = each thread copies its
 *                  own 16-byte vectors (cp.async) into a private ring, the
 *                  only form for rows split over a cluster; 0 = automatic
 *                  (2 where available, else 1).  A call asking for 2 where
 *                  it is not available takes 1.  The cross-entropy subset
 *                  always takes 1.  The two rings group the
 *                  first pass's partial sums differently, so (as with
 *                  ctas_per_row) results can differ in the last bits between
 *                  them; compare a forward with a backward or single launch
 *                  of the same ring.
 *   reserved     : must be 0.
 */
typedef struct {
  int32_t ctas_per_row;
  int32_t l2_keep;
  float stagger;
  int32_t ring;
  int32_t reserved[4];
} fct_options;

/*
 * Forward of the fused loss (PR #1384 analysis, "Forward Pass": step 1 is the
 * per-row log-sum-exp of student and teacher, step 2 the TVD and sigma
 * reductions, closed by the five per-row stores).
 *
 *   student, teacher : (BT, V) logits, element type `dtype`, strides ld_*.
 *   target           : (BT,) int64.
 *   ce, tvd, student_lse, teacher_lse, sigma : (BT,) fp32 outputs; none may
 *                      overlap another output or an input.
 *
 * The saved state needed by the backward is student_lse, teacher_lse and
 * sigma (O(BT)); no (BT, V) buffer is written.
 */
int fused_ce_tvd_forward(const void* student, int64_t ld_student,
                         const void* teacher, int64_t ld_teacher,
                         fct_dtype dtype, const int64_t* target, int64_t BT,
                         int64_t V, int64_t ignore_index, float* ce,
                         float* tvd, float* student_lse, float* teacher_lse,
                         float* sigma, int32_t* dev_status, void* stream);
int fused_ce_tvd_forward_ex(const void* student, int64_t ld_student,
                            const void* teacher, int64_t ld_teacher,
                            fct_dtype dtype, const int64_t* target, int64_t BT,
                            int64_t V, int64_t ignore_index, float* ce,
                            float* tvd, float* student_lse, float* teacher_lse,
                            float* sigma, const fct_options* options,
                            int32_t* dev_status, void* stream);

/*
 * Backward of the fused loss (PR #1384 analysis, "Backward Pass": reload the
 * student and teacher rows, recompute p, q and the sign from the saved lse
 * values, and combine both terms with the saved sigma).
 *
 *   student_lse, teacher_lse, sigma : (BT,) fp32, as written by
 *                      fused_ce_tvd_forward for the same logits.
 *   grad_ce, grad_tvd : upstream gradients; grad_stride = 1 reads BT values,
 *                      grad_stride = 0 broadcasts element 0 to every row.
 *   grad_student     : (BT, V) output, element type `dtype`, stride ld_grad.
 *                      grad_student == student with ld_grad == ld_student
 *                      computes the gradient IN PLACE over the student
 *                      logits; any other overlap with an input is
 *                      FCT_ERR_INVALID_ARG.
 *
 * bf16 gradients are rounded once, to nearest even, from fp32.
 */
int fused_ce_tvd_backward(const void* student, int64_t ld_student,
                          const void* teacher, int64_t ld_teacher,
                          fct_dtype dtype, const int64_t* target, int64_t BT,
                          int64_t V, int64_t ignore_index,
                          const float* student_lse, const float* teacher_lse,
                          const float* sigma, const float* grad_ce,
                          const float* grad_tvd, int64_t grad_stride,
                          void* grad_student, int64_t ld_grad,
                          int32_t* dev_status, void* stream);

/*
 * Forward and backward with sign words.  The "Backward Pass" reloads student
 * and teacher to recompute p, q and sign(p - q).  These two calls let the
 * forward keep the one piece of the teacher the backward needs, the sign of
 * p_v - q_v, as one bit per element, so the backward reads the student and
 * the bits (about V/8 bytes per row) instead of the teacher.  At 8192 x
 * 151936 bf16 that is 5.1 GB of backward traffic instead of 7.5 GB.  The
 * outputs are bit-identical to fused_ce_tvd_forward / fused_ce_tvd_backward.
 *
 *   signs    : (BT, ld_signs) bytes, written by the forward and read by the
 *              backward.  Per row: a uint32 tie flag, then one byte of sign
 *              bits per 16-byte vector of the row (element j of the vector at
 *              bit VEC-1-j, 1 where p < q).  ld_signs >=
 *              fused_ce_tvd_signs_row_bytes(V, dtype) and a multiple of 4;
 *              4-byte aligned.
 *   teacher  : still required by the backward.  A row with an exact tie
 *              (sign 0 somewhere), and the ragged tail of every row (V not a
 *              multiple of the vector), recompute their signs from it, and
 *              so does a whole call whose rows are not 16-byte aligned (the
 *              forward then sets every row's tie flag).
 * All other arguments are as for fused_ce_tvd_forward / fused_ce_tvd_backward.
 */
int64_t fused_ce_tvd_signs_row_bytes(int64_t V, fct_dtype dtype);

int fused_ce_tvd_forward_signs(const void* student, int64_t ld_student,
                               const void* teacher, int64_t ld_teacher,
                               fct_dtype dtype, const int64_t* target,
                               int64_t BT, int64_t V, int64_t ignore_index,
                               float* ce, float* tvd, float* student_lse,
                               float* teacher_lse, float* sigma,
                               uint8_t* signs, int64_t ld_signs,
                               int32_t* dev_status, void* stream);
int fused_ce_tvd_forward_signs_ex(const void* student, int64_t ld_student,
                                  const void* teacher, int64_t ld_teacher,
                                  fct_dtype dtype, const int64_t* target,
                                  int64_t BT, int64_t V, int64_t ignore_index,
                                  float* ce, float* tvd, float* student_lse,
                                  float* teacher_lse, float* sigma,
                                  uint8_t* signs, int64_t ld_signs,
                                  const fct_options* options,
                                  int32_t* dev_status, void* stream);

int fused_ce_tvd_backward_signs(const void* student, int64_t ld_student,
                                const void* teacher, int64_t ld_teacher,
                                fct_dtype dtype, const int64_t* target,
                                int64_t BT, int64_t V, int64_t ignore_index,
                                const float* student_lse,
                                const float* teacher_lse, const float* sigma,
                                const uint8_t* signs, int64_t ld_signs,
                                const float* grad_ce, const float* grad_tvd,
                                int64_t grad_stride, void* grad_student,
                                int64_t ld_grad, int32_t* dev_status,
                                void* stream);

/*
 * Forward and backward in ONE launch, for callers that know the upstream
 * gradients before the forward (for instance a mean over tokens, whose
 * per-row gradients are constants).  Writes everything
 * fused_ce_tvd_forward writes and the gradient fused_ce_tvd_backward would
 * write, bit for bit, but reads each logit from HBM once instead of twice:
 * the row stays in L2 for a third pass that applies the "Backward Pass"
 * formula with the row's sigma (PR #1384 analysis; fusing the two kernels is
 * this library's addition).
 *
 *   grad_ce, grad_tvd, grad_stride : as for fused_ce_tvd_backward.
 *   ce ... sigma : (BT,) fp32 outputs, as for fused_ce_tvd_forward.
 *   grad_student : (BT, V) output; grad_student == student (same ld) is in
 *                  place.  Rows that are not 16-byte aligned fall back to the
 *                  two launches (same results).
 */
int fused_ce_tvd_forward_backward(const void* student, int64_t ld_student,
                                  const void* teacher, int64_t ld_teacher,
                                  fct_dtype dtype, const int64_t* target,
                                  int64_t BT, int64_t V, int64_t ignore_index,
                                  const float* grad_ce, const float* grad_tvd,
                                  int64_t grad_stride, float* ce, float* tvd,
                                  float* student_lse, float* teacher_lse,
                                  float* sigma, void* grad_student,
                                  int64_t ld_grad, int32_t* dev_status,
                                  void* stream);
int fused_ce_tvd_forward_backward_ex(
    const void* student, int64_t ld_student, const void* teacher,
    int64_t ld_teacher, fct_dtype dtype, const int64_t* target, int64_t BT,
    int64_t V, int64_t ignore_index, const float* grad_ce,
    const float* grad_tvd, int64_t grad_stride, float* ce, float* tvd,
    float* student_lse, float* teacher_lse, float* sigma, void* grad_student,
    int64_t ld_grad, const fct_options* options, int32_t* dev_status,
    void* stream);

/*
 * The single launch above with its inputs and outputs in HOST memory, end to
 * end: row blocks of block_rows rows are copied to the device, computed, and
 * their gradient and per-row outputs copied back, with the copies of later
 * blocks overlapping the compute of earlier ones (PR #1384 analysis: the
 * "Forward Pass" and "Backward Pass" of the loss; streaming it from and to
 * host memory is this library's addition).  The results equal
 * fused_ce_tvd_forward_backward on the same rows, bit for bit.
 *
 *   student, teacher, target, grad_ce, grad_tvd : HOST inputs, laid out as
 *                  for fused_ce_tvd_forward_backward.
 *   ce, tvd, student_lse, teacher_lse, sigma : HOST outputs of BT floats, or
 *                  NULL (not returned).
 *   grad_student : HOST output (BT, V) with row stride ld_grad, or NULL.
 *                  Host outputs must not overlap the host inputs.
 *   workspace    : DEVICE memory of fused_ce_tvd_host_workspace_size(V,
 *                  dtype, min(block_rows, BT)) bytes, 256-byte aligned,
 *                  clobbered: a ring of three slots, each holding a block of
 *                  student and teacher logits (the gradient is computed in
 *                  place over the student block) and its per-row vectors.
 *   status       : HOST int32 or NULL; receives the OR of the device status
 *                  bits (FCT_DEV_*) of all blocks once `stream` reaches the
 *                  end of this call's work.
 *   stream       : the caller's stream; the kernels run on it, and the copies
 *                  on two streams of this call that are ordered after the
 *                  caller's earlier work on `stream` and joined back into it
 *                  before the call returns (later work on `stream` sees every
 *                  output).  The streams and events are created and released
 *                  by each call.
 *
 * The host buffers must be page-locked (cudaHostAlloc or cudaHostRegister)
 * for the copies to run asynchronously and overlap the compute; with
 * pageable memory the results are the same but the copies serialise.  Read
 * the host outputs only after synchronising `stream`.  BT == 0 returns
 * FCT_OK and writes nothing.  A block_rows or V beyond the supported range
 * (V > 2^40, block_rows > 2^20) returns FCT_ERR_UNSUPPORTED, as does the
 * workspace query (0).
 */
size_t fused_ce_tvd_host_workspace_size(int64_t V, fct_dtype dtype,
                                        int64_t block_rows);

int fused_ce_tvd_forward_backward_host(
    const void* student, int64_t ld_student, const void* teacher,
    int64_t ld_teacher, fct_dtype dtype, const int64_t* target, int64_t BT,
    int64_t V, int64_t ignore_index, const float* grad_ce,
    const float* grad_tvd, int64_t grad_stride, float* ce, float* tvd,
    float* student_lse, float* teacher_lse, float* sigma, void* grad_student,
    int64_t ld_grad, void* workspace, size_t workspace_bytes,
    int64_t block_rows, int32_t* status, void* stream);

/*
 * Fused-linear CE + TVD: the loss from hidden states and lm_head weights,
 * without ever holding the (BT, V) logits.  Rows go through in blocks of
 * chunk_rows: per block, the library's tensor-core GEMMs (fct_gemm_bf16:
 * bf16 in, fp32 accumulate) write the block's student and teacher logits
 * into `workspace`, the single-launch
 * forward + backward of the PR #1384 analysis's loss runs on them and writes
 * their logit gradient as bf16 (also in `workspace`), and two more GEMMs
 * give d loss / d h_student for the block and accumulate d loss / d
 * w_student.
 * (Computing logits in row blocks is the chunking that the Liger-Kernel
 * overview page describes for its fused linear cross-entropy; applying it to
 * CE + TVD is this library's addition.)  The teacher is frozen.
 *
 *   h_student (BT, d_student), w_student (V, d_student),
 *   h_teacher (BT, d_teacher), w_teacher (V, d_teacher): bf16, row strides
 *                    ld_*; 16-byte aligned with ld_* multiples of 8 (the
 *                    GEMMs' tile loads are TMA copies), else
 *                    FCT_ERR_ALIGNMENT (the no-allocation variant below
 *                    accepts any layout).
 *   target, grad_ce, grad_tvd, grad_stride, ce ... sigma: as for
 *                    fused_ce_tvd_forward_backward.
 *   grad_h_student : (BT, d_student) bf16 output, or NULL.
 *   grad_w_student : (V, d_student) fp32, ACCUMULATED into (+=), or NULL.
 *   logits_dtype   : element type of the logit blocks the loss sees.
 *                    FCT_F32: the GEMMs' fp32 sums of bf16 products, the
 *                    logit gradient rounded to bf16 into its own region.
 *                    FCT_BF16: those sums rounded once to bf16 (what a bf16
 *                    model's lm_head outputs, and the element type of the
 *                    analysis's V = 151936 workload); half the block bytes,
 *                    and the bf16 gradient overwrites the student block.
 *                    Anything else: FCT_ERR_UNSUPPORTED.
 *   workspace      : device memory of fused_linear_ce_tvd_workspace_size(V,
 *                    chunk_rows, logits_dtype) bytes, 256-byte aligned;
 *                    clobbered.  It holds the logit blocks and two blocks'
 *                    logit gradients: d w_student is accumulated once per two
 *                    row blocks (one read-modify-write of the fp32 (V, d)
 *                    matrix per 2 * chunk_rows rows).
 *                    fused_linear_ce_tvd_workspace_size returns 0 for V <= 0,
 *                    chunk_rows <= 0, an unknown dtype or a size that does
 *                    not fit a size_t.
 * V, d_*, the row strides and 2 * chunk_rows are GEMM dimensions: at most
 * 2^31 - 1024 each, else FCT_ERR_UNSUPPORTED.
 * The logits GEMMs' epilogue also writes each row's log-sum-exp as base-2
 * (max, sum) states per 256 logit columns (in the workspace), so the loss
 * kernel takes step 1 of "Forward Pass" from those states and reads each
 * logit block twice instead of three times.  The d hidden GEMM (few output
 * tiles, K = V) may split K, with its fp32 partial sums in the teacher block
 * of the workspace, which the loss has finished reading by then.
 */
size_t fused_linear_ce_tvd_workspace_size(int64_t V, int64_t chunk_rows,
                                          fct_dtype logits_dtype);

int fused_linear_ce_tvd_forward_backward(
    const void* h_student, int64_t ld_h_student, const void* w_student,
    int64_t ld_w_student, int64_t d_student, const void* h_teacher,
    int64_t ld_h_teacher, const void* w_teacher, int64_t ld_w_teacher,
    int64_t d_teacher, const int64_t* target, int64_t BT, int64_t V,
    int64_t ignore_index, const float* grad_ce, const float* grad_tvd,
    int64_t grad_stride, float* ce, float* tvd, float* student_lse,
    float* teacher_lse, float* sigma, void* grad_h_student, int64_t ld_grad_h,
    float* grad_w_student, int64_t ld_grad_w, fct_dtype logits_dtype,
    void* workspace, size_t workspace_bytes, int64_t chunk_rows,
    int32_t* dev_status, void* stream);

/*
 * Fused-linear CE + TVD that allocates nothing (no counterpart in the PR
 * #1384 analysis or the Liger-Kernel pages: it only changes where the
 * temporary logit blocks live).
 *
 * Some callers cannot let a library allocate device memory while they run:
 * processes whose memory is fixed up front (a caching allocator or a KV
 * cache that owns all free HBM, where a cudaMalloc outside it fails or
 * fragments it) and code that must not synchronise the device, which
 * cudaMalloc and cudaFree may do.  The entry point above needs a caller
 * workspace.  This one takes
 * the same arguments minus logits_dtype, workspace, workspace_bytes and
 * chunk_rows, and computes the outputs of the entry point above with
 * logits_dtype = FCT_F32, with:
 *   - its logit blocks in a fixed array of FCT_NOALLOC_SCRATCH_BYTES
 *     (64 MiB) of device memory that belongs to the library (a file-scope
 *     __device__ array): the driver reserves it on each device when the
 *     library's module holding it is loaded there and keeps it until the
 *     process exits;
 *   - its GEMMs on the library's tensor-core GEMM (fct_gemm_bf16, without
 *     a K split) when h_* and w_* have 16-byte aligned rows (ld a multiple
 *     of 8), else on a tiled CUDA-core kernel of the library (fp32
 *     accumulation; much slower at large sizes), so unaligned layouts are
 *     accepted here;
 *   - the same loss kernel and the same bf16 rounding of the logit gradient.
 * Rows go through in blocks of FCT_NOALLOC_SCRATCH_BYTES /
 * (8 * round_up(V, 8)) rows.  V up to 8,388,608 is supported; a larger V
 * (one student + teacher fp32 row would not fit) returns
 * FCT_ERR_UNSUPPORTED before any launch.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and queries the
 * device; make that first call before any stream capture.  Every call
 * shares the one array and leaves its last contents there; nothing in it
 * needs to start at zero (each block writes its logits before reading
 * them).  Calls whose work can overlap on the GPU (other streams, other host
 * threads) race on the array and give wrong results; order them.
 */
#define FCT_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

int fused_linear_ce_tvd_forward_backward_noalloc(
    const void* h_student, int64_t ld_h_student, const void* w_student,
    int64_t ld_w_student, int64_t d_student, const void* h_teacher,
    int64_t ld_h_teacher, const void* w_teacher, int64_t ld_w_teacher,
    int64_t d_teacher, const int64_t* target, int64_t BT, int64_t V,
    int64_t ignore_index, const float* grad_ce, const float* grad_tvd,
    int64_t grad_stride, float* ce, float* tvd, float* student_lse,
    float* teacher_lse, float* sigma, void* grad_h_student, int64_t ld_grad_h,
    float* grad_w_student, int64_t ld_grad_w, int32_t* dev_status,
    void* stream);

/*
 * The bf16 GEMM that the fused-linear entry point above runs its four
 * products on (logits = H W^T, d hidden = G W, d weight += G^T H; the
 * Liger-Kernel overview's fused linear cross-entropy computes the logits of
 * a row block by such a product and never holds the whole logit matrix),
 * exported as an operation of its own.  Hand-written for sm_103a: TMA tile
 * loads, tcgen05.mma with the accumulator in tensor memory, one persistent
 * CTA per SM.
 *
 *   C(m, n)  = sum_k A(m, k) B(n, k)   c_kind FCT_GEMM_F32 (fp32 C) or
 *                                      FCT_GEMM_BF16 (bf16 C, the fp32 sum
 *                                      rounded to nearest even);
 *   C(m, n) += sum_k A(m, k) B(n, k)   c_kind FCT_GEMM_ADD_F32 (fp32 C).
 *   Anything else: FCT_ERR_UNSUPPORTED.
 *
 *   A (M x K), B (N x K): bf16.  a_mn_major = 0: A(m, k) at A[m * lda + k]
 *            (K contiguous); 1: A(m, k) at A[k * lda + m] (M contiguous).
 *            Likewise b_mn_major for B.  Other values: FCT_ERR_INVALID_ARG.
 *            Both 16-byte aligned with lda, ldb multiples of 8 (the tile
 *            loads are TMA copies), else FCT_ERR_ALIGNMENT; lda, ldb at
 *            least the contiguous extent, else FCT_ERR_INVALID_ARG.
 *   C        : row-major M x N, row stride ldc >= N, aligned to its element;
 *            must not overlap A or B (FCT_ERR_INVALID_ARG).
 *   M, N >= 0 (0: nothing to do, FCT_OK), K >= 1; M, N, K at most
 *            2^31 - 1024, else FCT_ERR_UNSUPPORTED.
 *   workspace, workspace_bytes: optional (NULL, 0) device memory, 16-byte
 *            aligned, not overlapping A, B or C.  With it, a product whose
 *            output tiles (256 x 256) are too few to keep every SM pair
 *            busy and whose K is long may split K into parts: each part's
 *            fp32 partial sums go to the workspace and a second kernel adds
 *            them in part order (c_kind FCT_GEMM_F32 and FCT_GEMM_BF16
 *            only).  fct_gemm_bf16_workspace_size(M, N) bytes let every
 *            split happen; fewer allow fewer parts.
 * The tensor cores accumulate in fp32, K in blocks of 16 in increasing
 * order.  Without a split every element goes through the same sequence of
 * instructions, so a result depends only on its row of A and its row of B
 * (not on M, N or the tile it falls in); with one, also on the number of
 * parts, which is fixed by M, N, K, the workspace size and the device.
 * Repeated calls give identical bits either way.  Sums of products that are
 * exact in fp32 are exact.
 * dev_status (optional): FCT_DEV_WAIT_TIMEOUT is ORed in if
 * a pipeline wait in the kernel ran out (C is then invalid).
 */
#define FCT_GEMM_F32 0
#define FCT_GEMM_BF16 1
#define FCT_GEMM_ADD_F32 2

int fct_gemm_bf16(const void* A, int64_t lda, int32_t a_mn_major,
                  const void* B, int64_t ldb, int32_t b_mn_major, void* C,
                  int64_t ldc, int32_t c_kind, int64_t M, int64_t N, int64_t K,
                  void* workspace, size_t workspace_bytes, int32_t* dev_status,
                  void* stream);
/* Bytes of workspace for every K split of an M x N product; 0 for M or N
 * outside [1, 2^31) or a size that does not fit a size_t. */
size_t fct_gemm_bf16_workspace_size(int64_t M, int64_t N);

/*
 * Cross-entropy alone: the CE half of "Forward Pass" (one log-sum-exp pass,
 * ce = lse - logits[target]).  ce, lse: (BT,) fp32 outputs.
 */
int ce_forward(const void* logits, int64_t ld, fct_dtype dtype,
               const int64_t* target, int64_t BT, int64_t V,
               int64_t ignore_index, float* ce, float* lse,
               int32_t* dev_status, void* stream);
int ce_forward_ex(const void* logits, int64_t ld, fct_dtype dtype,
                  const int64_t* target, int64_t BT, int64_t V,
                  int64_t ignore_index, float* ce, float* lse,
                  const fct_options* options, int32_t* dev_status,
                  void* stream);

/*
 * Cross-entropy gradient alone: grad_ce*(p_v - 1[v==target]), the first of
 * the "Backward Pass" identities.  grad_logits may equal logits (with
 * ld_grad == ld) for an in-place gradient.
 */
int ce_backward(const void* logits, int64_t ld, fct_dtype dtype,
                const int64_t* target, int64_t BT, int64_t V,
                int64_t ignore_index, const float* lse, const float* grad_ce,
                int64_t grad_stride, void* grad_logits, int64_t ld_grad,
                int32_t* dev_status, void* stream);

/*
 * Cross-entropy forward and backward in one launch, given grad_ce: the
 * single-launch idea applied to the CE subset.  The row is read from HBM once
 * for its log-sum-exp and again from L2 for grad_ce*(p_v - 1[v==target]), so
 * HBM sees 1 read and 1 write per element instead of 2 reads and 1 write.
 * Outputs (ce, lse, grad_logits) are bit-identical to ce_forward followed by
 * ce_backward; grad_logits may equal logits (with ld_grad == ld) for an
 * in-place gradient.  Rows that are not 16-byte aligned take those two
 * launches.
 */
int ce_forward_backward(const void* logits, int64_t ld, fct_dtype dtype,
                        const int64_t* target, int64_t BT, int64_t V,
                        int64_t ignore_index, const float* grad_ce,
                        int64_t grad_stride, float* ce, float* lse,
                        void* grad_logits, int64_t ld_grad,
                        int32_t* dev_status, void* stream);
int ce_forward_backward_ex(const void* logits, int64_t ld, fct_dtype dtype,
                           const int64_t* target, int64_t BT, int64_t V,
                           int64_t ignore_index, const float* grad_ce,
                           int64_t grad_stride, float* ce, float* lse,
                           void* grad_logits, int64_t ld_grad,
                           const fct_options* options, int32_t* dev_status,
                           void* stream);

/*
 * Mean over tokens.  The method stores per-row ce and tvd and takes per-row
 * upstream gradients (PR #1384 analysis, "Forward Pass" stores and "Backward
 * Pass" combine); the reduction to a scalar is the caller's.  These give the
 * usual one, loss = (alpha * sum_r ce_r + beta * sum_r tvd_r) / n, with n the
 * number of rows whose target is not ignore_index (ignored rows have
 * ce = tvd = 0).  Each is one single-CTA launch with a fixed summation order
 * (fp64 accumulation), so results are deterministic.
 *
 * fused_ce_tvd_mean_upstream: from the targets alone (call it before the
 *   forward), writes grad_ce[0] = alpha / n and grad_tvd[0] = beta / n (0
 *   when n = 0), to pass with grad_stride = 0 to fused_ce_tvd_backward or
 *   fused_ce_tvd_forward_backward; *count = n if count is not NULL.
 * fused_ce_tvd_mean_loss: loss[0] from the forward's ce and tvd.
 * All pointers are device pointers; BT == 0 gives n = 0.
 */
int fused_ce_tvd_mean_upstream(const int64_t* target, int64_t BT,
                               int64_t ignore_index, double alpha, double beta,
                               float* grad_ce, float* grad_tvd, int64_t* count,
                               void* stream);
int fused_ce_tvd_mean_loss(const float* ce, const float* tvd,
                           const int64_t* target, int64_t BT,
                           int64_t ignore_index, double alpha, double beta,
                           float* loss, void* stream);

/*
 * Vocabulary-parallel split: the loss when the vocabulary is divided into
 * column ranges ("shards") across devices, each holding every row's columns
 * [v_begin, v_begin + V_shard) of the student and teacher logits.  A row's
 * log-sum-exp, TVD and sigma are sums over the vocabulary (PR #1384
 * analysis, "Forward Pass" steps 1 and 2; "Backward Pass"), so they split
 * into per-shard partials and a merge; distributing a model's vocabulary
 * this way is this library's addition.  One step, on every shard:
 *
 *   1. fused_ce_tvd_vp_lse          -> this shard's part1 (BT, 3)
 *   2. exchange: every device gathers all shards' part1 into
 *      parts1 (n_shards, BT, 3), in shard order (an all-gather)
 *   3. fused_ce_tvd_vp_merge_lse    -> ce, student_lse, teacher_lse (BT,)
 *   4. fused_ce_tvd_vp_tvd          -> this shard's part2 (BT, 2)
 *   5. exchange: parts2 (n_shards, BT, 2), in shard order
 *   6. fused_ce_tvd_vp_merge_tvd    -> tvd, sigma (BT,)
 *   7. fused_ce_tvd_vp_backward     -> the gradient of this shard's columns
 *
 * The merges fold the shards in shard order, so every device computes
 * bit-identical per-row values from the same gathered partials.  Only
 * 5 floats per row and shard cross devices.  Conventions as above, with:
 *
 *   student, teacher : the shard's first column of row 0 (row stride ld_*,
 *                      in elements, >= V_shard).
 *   target           : (BT,) int64 indices into the full vocabulary of V
 *                      entries; a target in another shard contributes no
 *                      -grad_ce term to this shard's gradient, and only a
 *                      target outside [0, V) (not ignore_index) is out of
 *                      range: the merge then writes NaN ce and sets
 *                      FCT_DEV_TARGET_OUT_OF_RANGE, and every shard's
 *                      backward writes that row's gradient as NaN.
 *   part (pass 1)    : (BT, 3) fp32: the shard's student lse, teacher lse,
 *                      and the student logit at the target when this shard
 *                      holds it (0 otherwise).  Ignored rows: zeros.
 *   part (pass 2)    : (BT, 2) fp32: the shard's sum of p*sign(p - q) and of
 *                      q*sign(p - q), p and q from the merged lse values.
 *   parts            : the n_shards partials stacked (shard k at k * BT rows).
 *   ce ... sigma     : as written by fused_ce_tvd_forward; ignored rows 0.
 *   grad_student     : the shard's (BT, V_shard) gradient columns; in place
 *                      over the shard's student columns when equal (same ld).
 */
int fused_ce_tvd_vp_lse(const void* student, int64_t ld_student,
                        const void* teacher, int64_t ld_teacher,
                        fct_dtype dtype, const int64_t* target, int64_t BT,
                        int64_t V_shard, int64_t v_begin, int64_t ignore_index,
                        float* part, void* stream);
int fused_ce_tvd_vp_merge_lse(const float* parts, int64_t n_shards,
                              const int64_t* target, int64_t BT, int64_t V,
                              int64_t ignore_index, float* ce,
                              float* student_lse, float* teacher_lse,
                              int32_t* dev_status, void* stream);
int fused_ce_tvd_vp_tvd(const void* student, int64_t ld_student,
                        const void* teacher, int64_t ld_teacher,
                        fct_dtype dtype, const int64_t* target, int64_t BT,
                        int64_t V_shard, int64_t ignore_index,
                        const float* student_lse, const float* teacher_lse,
                        float* part, void* stream);
int fused_ce_tvd_vp_merge_tvd(const float* parts, int64_t n_shards,
                              const int64_t* target, int64_t BT,
                              int64_t ignore_index, float* tvd, float* sigma,
                              void* stream);
int fused_ce_tvd_vp_backward(const void* student, int64_t ld_student,
                             const void* teacher, int64_t ld_teacher,
                             fct_dtype dtype, const int64_t* target, int64_t BT,
                             int64_t V_shard, int64_t v_begin, int64_t V,
                             int64_t ignore_index, const float* student_lse,
                             const float* teacher_lse, const float* sigma,
                             const float* grad_ce, const float* grad_tvd,
                             int64_t grad_stride, void* grad_student,
                             int64_t ld_grad, int32_t* dev_status,
                             void* stream);

/* Human-readable name of a fct_status value (static storage). */
const char* fct_status_string(int status);

/* Library version as 10000*major + 100*minor + patch.  300 and later: the
 * fused-linear entry point and its workspace query take logits_dtype.  400
 * and later: tuning goes through fct_options on the _ex entry points (no
 * process-wide knob).  500 and later: fct_gemm_bf16 and its workspace query;
 * the fused-linear workspace also holds the log-sum-exp partials of the
 * logits GEMMs (query its size again). */
int fct_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FUSED_CE_TVD_H_ */
