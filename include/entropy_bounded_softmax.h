/*
 * entropy_bounded_softmax.h -- C ABI of the GB300 (sm_103a) entropy-bounded
 * softmax library, libcsoftmax.so.
 *
 * The operation is `constrained_softmax` as defined by "BURT-IMMA CUDA Kernel
 * API Reference", section 2.1 (Signature, Parameters table, Description steps
 * 1-4), with the error codes of section 5.1, the NaN/Inf policy of section 5.3
 * and the degradation rule of section 5.4.  For each row l of a row-major
 * [batch, num_classes] fp32 matrix:
 *
 *   1. p = softmax(l) (T = 1) and its entropy H = -sum p_i ln p_i (nats);
 *   2. if H <= entropy_bound, write p and report T = 1;
 *   3. otherwise bisect T on [t_min, min(1, t_max)] for exactly max_iter
 *      steps: mid = (lo + hi) / 2; H(mid) > entropy_bound moves hi to mid,
 *      otherwise lo moves to mid.  Temperatures above 1 are never searched
 *      because H is nondecreasing in T (section 2.1 step 4).  The
 *      midpoints are the exact dyadic points t_min + j (hi0 - t_min) / 2^K
 *      (K = max_iter) rounded once to fp32; for max_iter > 24, where fp32
 *      cannot resolve those points, every fp32 value of the interval.
 *      Since H is monotone the result is the largest such point whose H is
 *      within the bound (t_min if none).  By default the cluster kernel
 *      finds it from a bracket of grid points closed by safeguarded Newton
 *      steps, evaluating H only where needed (cs_options.strict halves the
 *      bracket one evaluation at a time, i.e. bisects).  The row-group
 *      kernel, whose rows are a few registers per lane, takes one
 *      Newton-placed point per round;
 *   4. write softmax(l / lo) and report T = lo.  If even lo = t_min violates
 *      the bound, the row still gets softmax(l / t_min), the lowest entropy
 *      reachable (section 5.4), and ENTROPY_OVERFLOW is raised.
 *
 * Arithmetic is fp32 with the exponential on the hardware ex2 unit; the
 * grid points are indexed by integers and evaluated in fp32.
 *
 * All functions are thread-safe.  No function allocates device memory per
 * call; the library's only device objects are two 32-bit words per GPU (the
 * error word and the word cs_get_error reads it through).
 */
#ifndef ENTROPY_BOUNDED_SOFTMAX_H
#define ENTROPY_BOUNDED_SOFTMAX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  0-7 keep the numbering of section 5.1 (enum BurtError);
 * 8-10 are new.  4 (spectral overflow) and 5 (capacity full) belong to other
 * kernels of that page and are never returned here. */
typedef int32_t cs_status;
#define CS_OK 0
#define CS_ERR_NAN_INPUT 1        /* a row held a NaN (asynchronous)        */
#define CS_ERR_INF_INPUT 2        /* a row held +-Inf (asynchronous)        */
#define CS_ERR_ENTROPY_OVERFLOW 3 /* bound unsatisfiable at t_min (async)   */
#define CS_ERR_DIM_MISMATCH 6     /* batch < 0, num_classes < 1, overflow   */
#define CS_ERR_OOM 7              /* row too long for the shared-memory plan */
#define CS_ERR_INVALID_ARG 8      /* null/overlapping pointers, bad params  */
#define CS_ERR_CUDA 9             /* a CUDA call failed (launch, attribute)  */
#define CS_ERR_TIMEOUT 10         /* a bounded device wait gave up (async)  */

/* Kernel variants (cs_options.variant, cs_plan.variant). */
#define CS_VARIANT_AUTO 0
#define CS_VARIANT_ROWGROUP 1 /* 1-32 lanes per row, row in registers      */
#define CS_VARIANT_CLUSTER 2  /* 1-16 CTAs per row, row in shared memory,
                                 partial sums exchanged over DSMEM; one CTA
                                 per row when the cluster size is 1        */
#define CS_VARIANT_FUSED 3    /* biencoder_attention: all three steps in
                                 one kernel, step 3 on the fp32 FMA pipes
                                 (param = lanes per query row, 0 = auto)  */

/* Largest num_classes the library accepts: a 16-CTA cluster holding the row
 * in shared memory. */
#define CS_MAX_NUM_CLASSES 850000

/* Largest seq_len cs_attention_softmax accepts: one CTA holding a row in
 * shared memory. */
#define CS_MAX_SEQ_LEN 57344

/* Launch options; an all-zero struct (or NULL) means "automatic". */
typedef struct cs_options {
    int32_t variant;   /* CS_VARIANT_AUTO, _ROWGROUP or _CLUSTER            */
    int32_t param;     /* rowgroup: lanes per row (1, 2, 4, 8, 16, 32);
                          cluster: CTAs per row (1..16); 0 = automatic      */
    int32_t threads;   /* cluster: threads per CTA (multiple of 32,
                          64..512); 0 = automatic                           */
    int32_t strict;    /* 1 = bisect (H evaluated at every midpoint, one
                          pass per halving); 0 = close the bracket from
                          Newton-placed evaluations (same result for
                          monotone H, fewer passes: up to 3 points per
                          round in the cluster kernel, one in the
                          row-group kernel)                                 */
    int32_t* evals_out; /* cs_constrained_softmax_ex only; optional device
                          pointer, [batch] int32: how many temperatures each
                          row's exponentials were evaluated at, i.e. the ex2
                          per class the row cost (the T = 1 pass, every
                          point of every search round, and the output pass;
                          0 for a NaN/Inf row in the row-group kernel, 1 in
                          the cluster kernel, whose T = 1 pass runs before
                          the row's code is known).  NULL: not recorded.
                          Must not overlap logits, out or t_out.  The other
                          operations reject a non-NULL value.            */
} cs_options;

/* What a launch of the given shape uses.  Filled by cs_plan_launch /
 * cs_plan_host. */
typedef struct cs_plan {
    int32_t variant;         /* CS_VARIANT_ROWGROUP or CS_VARIANT_CLUSTER   */
    int32_t lanes_per_row;   /* rowgroup: lanes that share one row          */
    int32_t elems_per_lane;  /* rowgroup: fp32 registers of row per lane    */
    int32_t cluster_size;    /* cluster: CTAs per row (1 = one CTA per row) */
    int32_t slice_len;       /* cluster: classes held by one CTA            */
    int32_t threads_per_cta;
    int32_t smem_bytes;      /* dynamic shared memory per CTA               */
    int32_t ctas_per_sm;     /* CTAs resident per SM by the plan's limits   */
    int64_t grid_ctas;       /* CTAs in the launch                          */
    int32_t staged_tensors;  /* tensors a CTA keeps in shared memory
                                (cluster forward: 1, the logits; cluster
                                backward: 2, p and grad_out, or 1, p alone,
                                with grad_out read again; attention row-CTA:
                                1; biencoder: 3, keys, values and a tile of
                                queries, or 2, keys and queries, when step 3
                                runs on the tensor cores); rowgroup: 0     */
    int32_t tensor_cores;    /* biencoder: 1 when attn . V runs as a second
                                kernel on the tensor cores (tcgen05.mma)  */
    int32_t fan_points;      /* cluster forward: temperatures evaluated in
                                the T = 1 pass to bracket the search before
                                its first round (launches of at most one
                                wave, bound > 0, not strict; the kernel
                                drops them when the grid has no room);
                                0 otherwise                                */
} cs_plan;

/*
 * cs_constrained_softmax -- section 2.1 `constrained_softmax`.
 *
 * logits   device pointer, [batch, num_classes] fp32, row-major, contiguous.
 *          Read only.  Any 4-byte alignment is accepted; 16-byte aligned
 *          rows (num_classes % 4 == 0 and an aligned base) take the 128-bit
 *          load and store path.
 * out      device pointer, [batch, num_classes] fp32, written completely.
 *          Must not overlap logits (the page declares both __restrict__).
 * batch    rows; 0 is a no-op that returns CS_OK.
 * num_classes  classes per row, 1..CS_MAX_NUM_CLASSES.
 * entropy_bound  bound on H in nats (page default 0.20).  Any non-NaN value;
 *          a negative bound is unsatisfiable, +inf disables the search.
 * t_min, t_max  search interval (page defaults 0.01 and 10.0).  t_min must
 *          be a normal float in (0, 2^64] and t_max >= t_min (t_max may be
 *          +inf).  (The cap keeps every temperature used at or below 2^64,
 *          where logits that lie more than about 8.8e29 below the row's
 *          maximum contribute exactly 0, as they do in exact arithmetic.)
 * max_iter bisection steps, 0..1024 (page default 20).
 * t_out    optional device pointer, [batch] fp32: the temperature each row
 *          used (1 when no search was needed, lo after a search, t_min when
 *          the bound is unsatisfiable, NaN for a row with NaN/Inf input).
 *          May be NULL; must not overlap logits or out.
 * stream   a cudaStream_t (NULL = the legacy default stream).
 *
 * Ownership: the caller owns every buffer; nothing is allocated.
 * Execution: asynchronous on `stream`; the call returns after the launch
 * and never synchronises.
 * Errors: argument problems return CS_ERR_DIM_MISMATCH / CS_ERR_INVALID_ARG /
 * CS_ERR_OOM before anything is launched; a failed launch returns
 * CS_ERR_CUDA.  Per-row conditions found on the device (NaN, Inf,
 * unsatisfiable bound, wait timeout) do not fail the call: the rows get the
 * section 5.3/5.4 treatment (NaN/Inf rows are all zeros) and the condition
 * is OR-ed into the device error word, read with cs_get_error.
 */
cs_status cs_constrained_softmax(const float* logits, float* out,
                                 int64_t batch, int32_t num_classes,
                                 float entropy_bound, float t_min, float t_max,
                                 int32_t max_iter, float* t_out, void* stream);

/*
 * Same operation with launch options (tests and benchmarks use them to run
 * every variant on every shape).  options may be NULL (automatic).
 * A variant that cannot hold the row returns CS_ERR_OOM (rowgroup: more than
 * 32 classes per lane; cluster: slice larger than a CTA's shared memory);
 * malformed options return CS_ERR_INVALID_ARG.
 */
cs_status cs_constrained_softmax_ex(const float* logits, float* out,
                                    int64_t batch, int32_t num_classes,
                                    float entropy_bound, float t_min,
                                    float t_max, int32_t max_iter,
                                    float* t_out, const cs_options* options,
                                    void* stream);

/*
 * cs_constrained_softmax_bf16 -- the same operation on bf16 logits: a
 * work-reducing input form of section 2.1's kernel that halves the bytes
 * read per class (2 instead of 4; the output stays fp32).  Each logit is promoted to fp32 on load, which is exact (a
 * bf16 value is an fp32 value whose low 16 bits are zero), and from there
 * the computation is the fp32 one: the result equals, bit for bit,
 * cs_constrained_softmax on the promoted logits.
 *
 * logits   device pointer, [batch, num_classes] bf16 bit patterns
 *          (uint16_t), row-major, contiguous, 2-byte aligned.  Rows whose
 *          groups of four classes are 8-byte aligned (num_classes % 4 == 0
 *          and an 8-byte aligned base) take the vector load path.
 * Every other argument, the ownership, execution and error behaviour are
 * those of cs_constrained_softmax (out is fp32 and must not overlap the
 * logits' 2 * batch * num_classes bytes).
 */
cs_status cs_constrained_softmax_bf16(const uint16_t* logits, float* out,
                                      int64_t batch, int32_t num_classes,
                                      float entropy_bound, float t_min,
                                      float t_max, int32_t max_iter,
                                      float* t_out, void* stream);

/* The same with launch options (as cs_constrained_softmax_ex). */
cs_status cs_constrained_softmax_bf16_ex(const uint16_t* logits, float* out,
                                         int64_t batch, int32_t num_classes,
                                         float entropy_bound, float t_min,
                                         float t_max, int32_t max_iter,
                                         float* t_out,
                                         const cs_options* options,
                                         void* stream);

/* Host-only argument check of cs_constrained_softmax_bf16 (no CUDA call). */
cs_status cs_check_args_bf16(const uint16_t* logits, const float* out,
                             int64_t batch, int32_t num_classes,
                             float entropy_bound, float t_min, float t_max,
                             int32_t max_iter, const float* t_out);

/*
 * Reads and clears the calling thread's current device's error word, then
 * synchronises `stream`.  *code_mask receives a bitmask of (1 << code) for
 * every asynchronous condition since the last call: CS_ERR_NAN_INPUT,
 * CS_ERR_INF_INPUT, CS_ERR_ENTROPY_OVERFLOW, CS_ERR_TIMEOUT.  The read and
 * the clear are one atomic exchange, made by a one-thread kernel on `stream`
 * after the work enqueued on it before this call.  The word is shared by
 * every launch on the device: a launch on another stream that runs
 * concurrently reports its bits either to this call or to the next one,
 * never to neither.  Calls from several host threads are serialised.  This is
 * the only function that synchronises.  Returns CS_ERR_INVALID_ARG for a
 * NULL code_mask, CS_ERR_CUDA when a CUDA call fails.
 */
cs_status cs_get_error(int32_t* code_mask, void* stream);

/* The plan cs_constrained_softmax_ex would launch on the current device
 * (queries device attributes; no launch).  options may be NULL. */
cs_status cs_plan_launch(int64_t batch, int32_t num_classes,
                         const cs_options* options, cs_plan* plan);

/* The same planning on given device limits, host-only (no CUDA call):
 * sm_count SMs, smem_per_block_optin bytes of dynamic shared memory per CTA,
 * smem_per_sm bytes per SM, max_cluster CTAs per cluster. */
cs_status cs_plan_host(int64_t batch, int32_t num_classes,
                       const cs_options* options, int32_t sm_count,
                       int32_t smem_per_block_optin, int32_t smem_per_sm,
                       int32_t max_cluster, cs_plan* plan);

/* Host-only argument check of cs_constrained_softmax (no CUDA call). */
cs_status cs_check_args(const float* logits, const float* out, int64_t batch,
                        int32_t num_classes, float entropy_bound, float t_min,
                        float t_max, int32_t max_iter, const float* t_out);

/*
 * cs_constrained_softmax_backward -- gradient of a loss with respect to the
 * logits of cs_constrained_softmax.  "BURT-IMMA CUDA Kernel API Reference",
 * section 6.3 (PyTorch Custom Op Integration), gives the backward as the
 * softmax Jacobian product p * (g - <g, p>); the forward's output is
 * softmax(l / T), so every derivative carries 1/T, which that section leaves
 * out and this function restores.  Per row:
 *
 *     grad_in = (1/T) p * (grad_out - <grad_out, p>)
 *
 * T is the grid point the search settles on, piecewise constant in the
 * logits: it adds no term of its own, and this is the exact gradient
 * wherever one exists (everywhere except where a search comparison flips).
 *
 * probs     device pointer, [batch, num_classes] fp32, row-major: the
 *           forward's out.  Read only.
 * grad_out  device pointer, [batch, num_classes] fp32: dLoss/dout.  Read
 *           only; may overlap probs.
 * t         device pointer, [batch] fp32: the forward's t_out.  A row whose
 *           T is not a positive finite number gets an all-zero gradient
 *           (the forward reports NaN for the rows section 5.3 zeroes, whose
 *           output does not depend on the logits).
 * grad_in   device pointer, [batch, num_classes] fp32: dLoss/dlogits,
 *           written completely.  May be the same pointer as probs or
 *           grad_out (computed in place); any other overlap with probs,
 *           grad_out or t returns CS_ERR_INVALID_ARG.
 * batch     rows; 0 is a no-op that returns CS_OK.
 * num_classes  classes per row, 1..CS_MAX_NUM_CLASSES.
 * stream    a cudaStream_t (NULL = the legacy default stream).
 *
 * Any 4-byte alignment is accepted; rows whose four tensors share 16-byte
 * alignment take 128-bit loads and stores.  Arithmetic is fp32: the dot
 * product is summed in fp32 (per-thread chains, then shuffle and slot
 * trees), 1/T is the correctly rounded reciprocal.  NaN or Inf in probs or
 * grad_out propagates by IEEE arithmetic through the row's dot product.
 * Ownership: the caller owns every buffer; nothing is allocated.
 * Execution: asynchronous on `stream`; never synchronises.
 * Errors: argument problems return CS_ERR_DIM_MISMATCH / CS_ERR_INVALID_ARG /
 * CS_ERR_OOM before anything is launched; a failed launch returns
 * CS_ERR_CUDA.  Nothing is written to the device error word.
 */
cs_status cs_constrained_softmax_backward(const float* probs,
                                          const float* grad_out,
                                          const float* t, float* grad_in,
                                          int64_t batch, int32_t num_classes,
                                          void* stream);

/*
 * Same with launch options (NULL = automatic): variant CS_VARIANT_ROWGROUP
 * (param = lanes per row, 1..32, a power of two; the row must fit 32
 * classes per lane, else CS_ERR_OOM) or CS_VARIANT_CLUSTER (param = CTAs per
 * row, 1..16; threads as for the forward).  strict must be 0.
 */
cs_status cs_constrained_softmax_backward_ex(const float* probs,
                                             const float* grad_out,
                                             const float* t, float* grad_in,
                                             int64_t batch,
                                             int32_t num_classes,
                                             const cs_options* options,
                                             void* stream);

/* The backward's launch plan on the current device (no launch), and the
 * same planning on given device limits, host-only (as cs_plan_host). */
cs_status cs_plan_backward_launch(int64_t batch, int32_t num_classes,
                                  const cs_options* options, cs_plan* plan);
cs_status cs_plan_backward_host(int64_t batch, int32_t num_classes,
                                const cs_options* options, int32_t sm_count,
                                int32_t smem_per_block_optin,
                                int32_t smem_per_sm, int32_t max_cluster,
                                cs_plan* plan);

/* Host-only argument check of cs_constrained_softmax_backward (no CUDA
 * call). */
cs_status cs_check_backward_args(const float* probs, const float* grad_out,
                                 const float* t, const float* grad_in,
                                 int64_t batch, int32_t num_classes);

/*
 * cs_attention_softmax -- section 2.6 `attention_softmax`.  For every row
 * (b, h, i) of the scores, with keys j = 0..seq_len-1:
 *
 *   1. v_j = scores[b, h, i, j] + mask[b, j], added in fp32 (mask NULL
 *      adds nothing); a mask value of -inf removes key j, and the page's
 *      -1e9 works as written (near 1e9 fp32 steps by 64);
 *   2. causal: keys j > i are removed and never read;
 *   3. out = softmax over the kept keys with the max subtracted (exp on the
 *      ex2 unit, fp32 sums); removed keys get exactly 0.
 *
 * scores   device pointer, [batch, heads, seq_len, seq_len] fp32,
 *          row-major.  Read only.
 * out      device pointer, same shape, written completely.  May be the same
 *          pointer as scores (in place, which section 2.6 allows); any
 *          other overlap returns CS_ERR_INVALID_ARG.
 * mask     device pointer, [batch, seq_len] fp32 (section 2.6's
 *          [batch, 1, 1, seq_len]), or NULL.  Read only; must not overlap
 *          out.
 * batch, heads, seq_len  >= 0 (no rows: a no-op returning CS_OK);
 *          seq_len <= CS_MAX_SEQ_LEN.
 * causal   0 or 1.
 * stream   a cudaStream_t (NULL = the legacy default stream).
 *
 * Any 4-byte alignment is accepted; rows that start 16-byte aligned (an
 * aligned base and seq_len % 4 == 0) take 128-bit loads and stores.
 * Section 5.3: a NaN or an infinity among the scores and mask values a row
 * uses (a mask of -inf excepted) zeroes that row and ORs CS_ERR_NAN_INPUT
 * (a NaN was seen) or CS_ERR_INF_INPUT into the error word (cs_get_error).
 * A row whose keys are all removed is written as zeros without a flag.
 * Ownership, execution and argument errors: as cs_constrained_softmax.
 */
cs_status cs_attention_softmax(const float* scores, float* out,
                               const float* mask, int32_t batch,
                               int32_t heads, int32_t seq_len,
                               int32_t causal, void* stream);

/*
 * Same with launch options (NULL = automatic): CS_VARIANT_ROWGROUP (param =
 * lanes per row, 1..32, a power of two; at most 32 scores per lane, else
 * CS_ERR_OOM) or CS_VARIANT_CLUSTER, which here means one CTA per row
 * (param 0 or 1; threads as for the forward).  strict must be 0.
 */
cs_status cs_attention_softmax_ex(const float* scores, float* out,
                                  const float* mask, int32_t batch,
                                  int32_t heads, int32_t seq_len,
                                  int32_t causal, const cs_options* options,
                                  void* stream);

/* The attention launch plan on the current device (no launch), and the
 * same planning on given device limits, host-only.  aligned = 1 when every
 * row starts 16-byte aligned (aligned scores and out, seq_len % 4 == 0),
 * which lets the row-group plan count float4s exactly. */
cs_status cs_plan_attention_launch(int32_t batch, int32_t heads,
                                   int32_t seq_len, int32_t aligned,
                                   const cs_options* options, cs_plan* plan);
cs_status cs_plan_attention_host(int32_t batch, int32_t heads,
                                 int32_t seq_len, int32_t aligned,
                                 const cs_options* options, int32_t sm_count,
                                 int32_t smem_per_block_optin,
                                 int32_t smem_per_sm, cs_plan* plan);

/* Host-only argument check of cs_attention_softmax (no CUDA call). */
cs_status cs_check_attention_args(const float* scores, const float* out,
                                  const float* mask, int32_t batch,
                                  int32_t heads, int32_t seq_len,
                                  int32_t causal);

/*
 * cs_biencoder_attention -- section 2.5 `biencoder_attention`, fused.  For
 * every batch b, head h and query i:
 *
 *   1. scores_j = (query_i . key_j) * scale, j < context_len.  The dot
 *      product is evaluated in fp32 as one fused multiply-add per d in
 *      order d = 0..d_head-1 from 0, then one fp32 multiply by scale: the
 *      page's kernel is fp32 and the search turns these logits into a grid
 *      point, so the evaluation is fixed rather than left to a GEMM's
 *      blocking;
 *   2. attn = constrained_softmax(scores, entropy_bound) per query row
 *      (cs_constrained_softmax's operation, including its NaN/Inf and
 *      unsatisfiable-bound policy and error bits);
 *   3. output_i = sum_j attn_j value_j.
 *
 * query    device pointer, [batch, num_heads, query_len, d_head] fp32.
 * context_keys, context_values  device pointers, [batch, num_heads,
 *          context_len, d_head] fp32.  All three read only.
 * output   device pointer, [batch, num_heads, query_len, d_head] fp32,
 *          written completely; must not overlap the inputs.
 * batch_size, query_len, num_heads >= 0 (no rows: a no-op returning CS_OK);
 * context_len 1..256; d_head 1..256 and a multiple of 4 (else
 *          CS_ERR_INVALID_ARG); larger shapes return CS_ERR_OOM.
 * scale    finite (the page passes 1/sqrt(d_head)).
 * entropy_bound  as for cs_constrained_softmax (page default 0.20); the
 *          search takes the section 2.1 defaults t_min 0.01, t_max 10.0,
 *          max_iter 20.
 * stream   a cudaStream_t (NULL = the legacy default stream).
 *
 * The four bases must be 16-byte aligned (float4 staging); otherwise
 * CS_ERR_INVALID_ARG.  Ownership, execution, errors: as
 * cs_constrained_softmax.
 *
 * Kernels.  For d_head <= 64 and context_len <= d_head (the page's shape),
 * steps 1 and 2 run in one kernel that writes the weights, and step 3
 * (attn @ context_values) runs in a second kernel on the tensor cores
 * (tcgen05.mma, TF32 operands, three TF32 products per fp32 product for
 * fp32 accuracy, fp32 accumulation in tensor memory).  The weights pass
 * through attn_out when it is given, otherwise through the output buffer
 * itself (the first context_len floats of each output row, overwritten by
 * the result): no scratch memory is used.  Other shapes, and
 * CS_VARIANT_FUSED, run all three steps in one kernel on the fp32 FMA
 * pipes, with nothing between the steps in global memory.
 */
cs_status cs_biencoder_attention(const float* query,
                                 const float* context_keys,
                                 const float* context_values, float* output,
                                 int32_t batch_size, int32_t query_len,
                                 int32_t context_len, int32_t d_head,
                                 int32_t num_heads, float scale,
                                 float entropy_bound, void* stream);

/*
 * The same with the search parameters of cs_constrained_softmax and two
 * optional outputs: attn_out [batch, num_heads, query_len, context_len]
 * (the weights of step 2) and t_out [batch, num_heads, query_len] (each
 * row's temperature), either may be NULL.  options: CS_VARIANT_AUTO,
 * CS_VARIANT_ROWGROUP with param = lanes per query row (a power of two,
 * 8 x lanes >= context_len), or CS_VARIANT_FUSED (one kernel; param as
 * for ROWGROUP, 0 = automatic); threads and strict must be 0.
 */
cs_status cs_biencoder_attention_ex(const float* query,
                                    const float* context_keys,
                                    const float* context_values,
                                    float* output, int32_t batch_size,
                                    int32_t query_len, int32_t context_len,
                                    int32_t d_head, int32_t num_heads,
                                    float scale, float entropy_bound,
                                    float t_min, float t_max,
                                    int32_t max_iter, float* attn_out,
                                    float* t_out, const cs_options* options,
                                    void* stream);

/* Host-only plan (lanes per query row, CTAs, shared memory) for the given
 * limits, and host-only argument check of cs_biencoder_attention_ex. */
cs_status cs_plan_biencoder_host(int32_t batch_size, int32_t query_len,
                                 int32_t context_len, int32_t d_head,
                                 int32_t num_heads, const cs_options* options,
                                 int32_t smem_per_block_optin, cs_plan* plan);
cs_status cs_check_biencoder_args(const float* query,
                                  const float* context_keys,
                                  const float* context_values,
                                  const float* output, int32_t batch_size,
                                  int32_t query_len, int32_t context_len,
                                  int32_t d_head, int32_t num_heads,
                                  float scale, float entropy_bound,
                                  float t_min, float t_max, int32_t max_iter,
                                  const float* attn_out, const float* t_out);

/*
 * Throughput probe of the ex2 unit, the unit this operation is bound by.
 * Launches one kernel over all SMs in which every thread runs `iters`
 * rounds of 8 independent ex2.approx.ftz.f32 chains; *ex2_count receives
 * the number of ex2 the launch executes.  The caller times the launch (for
 * example with CUDA events on `stream`).  sink: device pointer to at least
 * cs_probe_ex2_sink_floats() floats, written so that the work is not dead.
 */
cs_status cs_probe_ex2(float* sink, int32_t iters, int64_t* ex2_count,
                       void* stream);
int32_t cs_probe_ex2_sink_floats(void);

/*
 * Exercises the bounded device wait that every kernel uses: launches one
 * CTA that waits on a barrier nothing completes, for at most limit_ns
 * nanoseconds (1..10^10), then gives up and records CS_ERR_TIMEOUT in the
 * error word.  Used to test the timeout path without hanging anything.
 */
cs_status cs_test_wait_timeout(int64_t limit_ns, void* stream);

/* Library version string, e.g. "1.0.0 sm_103a". */
const char* cs_version(void);

/* Short English name of a status code. */
const char* cs_status_string(cs_status status);

#ifdef __cplusplus
}
#endif

#endif /* ENTROPY_BOUNDED_SOFTMAX_H */
