/*
 * zero_gb300.h -- C ABI of libzero_gb300.so: one ZeRO step over N simulated
 * data-parallel ranks whose buffers all live in the memory of one GPU.
 *
 * The step (the "ZeRO-Sharded Adam Step" problem page, section "The step"):
 *   1. reduce-scatter: rank i receives the mean over the N ranks' local
 *      gradients, for the indices of its shard only;
 *   2. rank i runs Adam/AdamW on its shard with its own m and v (and its fp32
 *      master weights in mixed precision);
 *   3. all-gather: every rank's parameter replica receives all updated shards.
 * Shard i is np.array_split(np.arange(n), N)[i] (same page, "The shards").
 * The three steps run fused in one pass over memory; the mean gradient is
 * never stored. Around that step: whole-tensor shards, gradient-norm clipping
 * and an accumulation factor (zero_grad_norm_sq, zero_step_ex), momentum SGD
 * as the optimizer (zero_step_sgd), ZeRO stage 3 (owner-only steps and
 * zero_gather), 25 MiB bucket streaming, host-memory gradients
 * (zero_step_from_host, zero_step_from_host_ex), the DDP mean (also from host
 * memory: ddp_allreduce_mean_from_host) and per-stage memory accounting.
 *
 * Conventions for every call:
 *  - Return value: ZERO_OK (0) or a negative ZERO_E* code. zero_strerror()
 *    names a code; zero_last_error() gives the calling thread's last message.
 *  - Sizes are int64_t element counts; byte counts are uint64_t.
 *  - `params`, `grads`: HOST arrays of N DEVICE pointers, each to n elements
 *    (float for ZERO_FP32, bf16 bit patterns (uint16) for ZERO_BF16_MIXED),
 *    at least naturally aligned. Buffers sharing one 16-byte phase (the usual
 *    case: separate allocations) take the 16-byte vector path; any other
 *    layout is still correct, on a slower 4-/2-byte path.
 *  - With n == 0 nothing is read or written and NULL buffer pointers are
 *    accepted (the host arrays of pointers must still be non-NULL).
 *  - The caller owns every device buffer. The library never allocates device
 *    memory; zero_init_states allocates only a small host handle.
 *  - Device work is queued on the caller's stream (zero_stream_t is a
 *    cudaStream_t; NULL is the legacy default stream) and runs
 *    asynchronously; argument errors are reported before anything is queued.
 *  - Calls on distinct state handles may come from different host threads.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *zero_stream_t; /* same type as cudaStream_t */
typedef struct CUevent_st *zero_event_t;   /* same type as cudaEvent_t */

/* Storage precision of the training state. */
enum {
  ZERO_FP32 = 0,       /* fp32 params and grads, fp32 m, v: 4+4+8 bytes/param */
  ZERO_BF16_MIXED = 1, /* bf16 params and grads, fp32 master, m, v: 2+2+12    */
  ZERO_FP64_EMU = 2    /* float64 course-emulation bookkeeping (memory only)  */
};

/* Status codes. */
enum {
  ZERO_OK = 0,
  ZERO_EINVAL = -1,    /* bad n, N, stage, precision, t, hyperparameter, range or NULL */
  ZERO_EALIGN = -2,    /* a pointer is not aligned to its element size */
  ZERO_ECUDA = -3,     /* a CUDA runtime call or kernel launch failed */
  ZERO_ETIMEDOUT = -4, /* zero_step_bucketed: work not finished by the deadline */
  ZERO_ENOMEM = -5     /* host allocation of a state handle failed */
};

#define ZERO_MAX_RANKS 64

typedef struct zero_states zero_states_t;

/* ---------------------------------------------------------------- shards -- */

/* Shard offsets a_0..a_N of [0, n) over N ranks, written to the host array
 * bounds[N+1]: a_i = i*q + min(i, r) with q = n / N, r = n % N, i.e. the
 * pieces of np.array_split(np.arange(n), N) ("ZeRO-Sharded Adam Step",
 * "The shards"). n < N is legal and gives empty shards.
 * Errors: EINVAL if n < 0, N < 1, or bounds is NULL. */
int zero_shard_bounds(int64_t n, int32_t N, int64_t *bounds);

/* ----------------------------------------------------------------- state -- */

/* Build the optimizer state of all N ranks ("ZeRO-Sharded Adam Step", "What to
 * implement": init_states gives every worker zero m and v of its shard's
 * size). State is stored flat in global index order: rank i's m, v (and
 * master) are elements [a_i, a_{i+1}) of the caller's n-element device
 * buffers m, v, master, so a shard is a pure index range.
 *   m, v        : device float[n], zeroed here (queued on `stream`). For
 *                 momentum SGD (zero_step_sgd) pass v = NULL: m is the
 *                 momentum buffer; for SGD without momentum m = v = NULL.
 *                 The AdamW steps reject a state without v.
 *   master      : ZERO_BF16_MIXED only: device float[n], set to master_init;
 *                 must be NULL for ZERO_FP32.
 *   master_init : ZERO_BF16_MIXED only: device float[n], the fp32 initial
 *                 weights (the replicas are expected to hold their bf16
 *                 round-to-nearest-even); NULL for ZERO_FP32.
 *   out         : receives a host handle; release it with zero_free_states.
 * The handle records the buffers; they must outlive it.
 * Errors: EINVAL (n < 0, N outside [1, ZERO_MAX_RANKS], precision not FP32 or
 * BF16_MIXED, NULL or extra pointer, v without m), EALIGN, ECUDA, ENOMEM. */
int zero_init_states(int64_t n, int32_t N, int32_t precision, float *m, float *v,
                     float *master, const float *master_init, zero_stream_t stream,
                     zero_states_t **out);

/* zero_init_states with caller-chosen shard bounds: `bounds` is a HOST array
 * of N+1 offsets rising from 0 to n (NULL: the np.array_split shards). Rank i
 * owns [bounds[i], bounds[i+1]); shards may be empty. The step's arithmetic
 * does not depend on the bounds, only which replica holds each shard's
 * authoritative fp32 parameter. Use zero_tensor_shard_bounds for shards of
 * whole tensors. Errors: as zero_init_states, plus EINVAL for bad bounds. */
int zero_init_states_ex(int64_t n, int32_t N, int32_t precision, float *m, float *v,
                        float *master, const float *master_init, const int64_t *bounds,
                        zero_stream_t stream, zero_states_t **out);

/* Shards of whole tensors ("ZeRO One: Sharding the Optimizer", "Sharding
 * Parameters"): the T tensors of the flat vector (HOST array numels[T], in
 * parameters() order) are split like indices in np.array_split -- rank i gets
 * tensors [i*q + min(i, r), (i+1)*q + min(i+1, r)) with q = T / N, r = T % N --
 * and bounds[N+1] (HOST) receives the element offsets of those tensors, so no
 * tensor is split. Errors: EINVAL (T < 0, N < 1, NULL, a negative size,
 * overflow). */
int zero_tensor_shard_bounds(const int64_t *numels, int64_t T, int32_t N, int64_t *bounds);

/* Release a handle (the caller's device buffers are untouched). NULL is a no-op. */
int zero_free_states(zero_states_t *st);

/* n, N and precision of a handle (any output pointer may be NULL). */
int zero_states_info(const zero_states_t *st, int64_t *n, int32_t *N, int32_t *precision);

/* Rank `rank`'s shard [lo, hi) and its views into m, v, master (NULL for a
 * buffer the state does not have: master in fp32, v or m for SGD). Errors: EINVAL for a NULL handle or a rank outside [0, N). */
int zero_state_view(const zero_states_t *st, int32_t rank, int64_t *lo, int64_t *hi,
                    float **m, float **v, float **master);

/* ------------------------------------------------------------------ step -- */

/* One ZeRO step at step number t (1-based) over all n parameters.
 * For every index j, with a the owner rank of j:
 *   g   = (((g_0[j] + g_1[j]) + ...) + g_{N-1}[j]) / N      fp32, rank order
 *   p   = params[a][j] (fp32) or master[j] (mixed)
 *   p   = p * fl(1 - lr*wd)                                  decoupled decay
 *   m   = fl(b1)*m + fl(1-b1)*g;   v = fl(b2)*v + fl(1-b2)*(g*g)
 *   p   = p - fl(lr/(1-b1^t)) * (m / (sqrt(v)/fl(sqrt(1-b2^t)) + fl(eps)))
 *   params[r][j] = p for every r (mixed: master[j] = p, params[r][j] = bf16 RNE(p))
 * Every operation is one IEEE fp32 operation (no contraction); fl(.) is a
 * constant formed in double on the host and rounded to float once. wd = 0 is
 * plain Adam. The Adam formula is not printed on the pages; this is the
 * reading of "Data parallelism and ZeRO stages 1 to 3", section 3 (m_hat = g,
 * sqrt(v_hat) = |g| at t = 1) with PyTorch-style decoupled decay.
 * params and grads must not overlap one another or the state buffers.
 * Errors: EINVAL (NULL pointer or entry, t < 1, betas outside [0,1),
 * non-finite or negative lr/eps, non-finite wd), EALIGN, ECUDA. */
int zero_step(void *const *params, const void *const *grads, zero_states_t *st, int64_t t,
              double lr, double beta1, double beta2, double eps, double weight_decay,
              zero_stream_t stream);

/* zero_step restricted to the indices [lo, hi) (0 <= lo <= hi <= n): the update
 * is elementwise, so the steps of a partition of [0, n) equal one full step
 * bit for bit. Errors: as zero_step, plus EINVAL for a bad range. */
int zero_step_range(void *const *params, const void *const *grads, zero_states_t *st,
                    int64_t t, double lr, double beta1, double beta2, double eps,
                    double weight_decay, int64_t lo, int64_t hi, zero_stream_t stream);

/* ----------------------------------------------- clipping, accumulation -- */

/* Squared global L2 norm of the mean gradient, ||(1/N) sum_r g_r||^2, written
 * to the DEVICE scalar *norm_sq (queued on `stream`). This is the first half
 * of sharded global-norm clipping ("Data parallelism and ZeRO stages 1 to 3",
 * "Going further": an all-reduce of the squared chunk norms before the step):
 * the float mean of every element (rank order, as in the step) is squared
 * without rounding error (split into a float product and its exact error) and
 * summed with compensation, so each partial is accurate to about double
 * precision; fixed chunks of 32,768 elements give partial sums in `scratch` (a
 * DEVICE buffer of at least zero_grad_norm_scratch_count doubles,
 * caller-owned, contents overwritten), which one block adds in a fixed order.
 * The result does not depend on the GPU's size and is bit-reproducible.
 * Errors: EINVAL (n < 0, N outside [1, ZERO_MAX_RANKS], bad precision, NULL,
 * scratch too small, overlapping buffers), EALIGN, ECUDA. */
int zero_grad_norm_scratch_count(int64_t n, int32_t precision, int64_t *count);
int zero_grad_norm_sq(const void *const *grads, int64_t n, int32_t N, int32_t precision,
                      double *scratch, int64_t scratch_count, double *norm_sq,
                      zero_stream_t stream);

/* zero_grad_norm_sq without caller-provided scratch. Some callers cannot
 * allocate device memory at all: a process that runs inside a fixed memory
 * pool frozen after start-up, code that must not call cudaMalloc because it
 * synchronizes the device and would stall the work in flight on other
 * streams, or a hook (a logger, a health check) that only borrows the
 * gradient buffers and has no allocator of its own. This entry point allocates
 * nothing: its partial sums live in an array of 65,536 doubles (512 KB) that
 * the library keeps on every GPU that loads it, until the process exits.
 * There is no counterpart on the pages; it computes exactly what
 * zero_grad_norm_sq computes, bit for bit.
 *   grads, n, N, precision, stream : as zero_grad_norm_sq.
 *   norm_sq : DEVICE scalar receiving ||(1/N) sum_r g_r||^2 (caller-owned).
 * The first call on a device, with that device current, looks up the device
 * address of the array (a host-side runtime call) and keeps it for the life
 * of the process; make that first call before any stream capture, and do not
 * use this entry point on a device after cudaDeviceReset (the kept address
 * would be stale). Every call shares the one array: calls whose work can
 * overlap on the GPU (other streams, other host threads) race and must be
 * ordered by the caller. No other entry point uses the array. Each call
 * writes every partial it reads, so nothing needs clearing between calls.
 * Errors: as zero_grad_norm_sq, plus EINVAL when n > ZERO_NOALLOC_MAX_N
 * (use zero_grad_norm_sq with your own scratch above that). */
#define ZERO_NOALLOC_MAX_N 2147450880LL /* 65,535 partials x 32,768 elements */
int zero_grad_norm_sq_noalloc(const void *const *grads, int64_t n, int32_t N, int32_t precision,
                              double *norm_sq, zero_stream_t stream);

/* Options of zero_step_ex. */
typedef struct zero_step_opts {
  int64_t t;             /* step number, >= 1 */
  double lr, beta1, beta2, eps, weight_decay;
  /* Multiplies the mean gradient: 1.0 leaves it as is; 1/k turns the sum of k
   * accumulated micro-batch gradients into their mean ("Data Parallelism &
   * ZeRO", "Two more things you'll actually hit"). Finite, > 0. */
  double grad_scale;
  /* > 0: clip the scaled mean gradient to this global L2 norm with the
   * coefficient min(1, max_grad_norm / (grad_scale * sqrt(*norm_sq) + 1e-6));
   * <= 0: no clipping. */
  double max_grad_norm;
  /* DEVICE scalar, required when clipping, ignored otherwise. Without
   * norm_scratch it is an INPUT: the squared norm from zero_grad_norm_sq on
   * the same gradients, read on the device when the step runs (no host
   * synchronisation). With norm_scratch it is an OUTPUT (see below). */
  const double *norm_sq;
  int64_t lo, hi;        /* index range of the step; hi < 0 means n */
  /* Nonzero: ZeRO stage 3 ("Data parallelism and ZeRO stages 1 to 3",
   * section 2, stage 3). The all-gather is left out: the new parameters are
   * written only into the owner's replica, over the owner's shard, and every
   * other replica element is left as it was (released). zero_gather brings the
   * replicas back to the full parameters. 0: the stage-1/2 step. */
  int32_t owner_only;
  /* NULL, or (when clipping) a DEVICE buffer of at least norm_scratch_count
   * >= zero_grad_norm_scratch_count(n) doubles, caller-owned, overwritten,
   * 8-byte aligned and disjoint from every other buffer of the call. Given,
   * the call computes the squared norm of the whole gradient [0, n) itself,
   * as zero_grad_norm_sq does on the same buffers (the same launches, so the
   * same bits), writes it to *norm_sq and clips with it; the step is chained
   * to the norm's launches as a programmatic dependent (it starts while they
   * finish and waits for the norm before reading it). The norm's last launch
   * also forms the clip multiplier once, into the scratch's last slot, where
   * the step reads it (the same value the step would form from *norm_sq). The
   * host-input step requires it when clipping. */
  double *norm_scratch;
  int64_t norm_scratch_count;
} zero_step_opts_t;

/* zero_step with the options above. The multiplier grad_scale * coefficient
 * is formed on the device in double and rounded to float once; the mean
 * gradient is multiplied by it (one IEEE fp32 multiply) before the update.
 * With grad_scale = 1 and no clipping the result equals zero_step bit for bit.
 * Errors: as zero_step_range, plus EINVAL for a bad grad_scale or
 * max_grad_norm, clipping without norm_sq, a norm_scratch that is too small
 * or overlaps another buffer; EALIGN for a misaligned norm_scratch or
 * norm_sq. */
int zero_step_ex(void *const *params, const void *const *grads, zero_states_t *st,
                 const zero_step_opts_t *opts, zero_stream_t stream);

/* Options of zero_step_sgd: momentum SGD as the optimizer of the step. The
 * pages name SGD beside AdamW as an elementwise optimizer that ZeRO wraps
 * unchanged ("Data parallelism and ZeRO stages 1 to 3", section 2, stage 1;
 * its tests step DDP with momentum SGD, section 4) without printing its
 * update; this follows torch.optim.SGD. */
typedef struct zero_sgd_opts {
  int64_t t;             /* step number, >= 1; at t = 1 the buffer starts as g */
  double lr;             /* finite, >= 0 */
  double momentum;       /* mu >= 0; 0 = plain SGD (no buffer) */
  double dampening;      /* the buffer update is mu*buf + (1 - dampening)*g */
  double weight_decay;   /* coupled: g <- g + weight_decay * p (0: none) */
  int32_t nesterov;      /* nonzero: direction g + mu*buf (needs mu > 0, dampening 0) */
  double grad_scale;     /* as zero_step_opts_t */
  double max_grad_norm;  /* as zero_step_opts_t */
  const double *norm_sq; /* as zero_step_opts_t */
  int64_t lo, hi;        /* index range of the step; hi < 0 means n */
  int32_t owner_only;    /* as zero_step_opts_t: ZeRO stage 3 */
  double *norm_scratch;  /* as zero_step_opts_t */
  int64_t norm_scratch_count;
} zero_sgd_opts_t;

/* The fused ZeRO step with momentum SGD on each shard: reduce-scatter-mean
 * (times the multiplier of zero_step_ex), then per element, in IEEE fp32 with
 * every operation rounded separately:
 *   g <- g + wd*p                     (wd != 0)
 *   buf <- g (t = 1), else mu*buf + (1 - dampening)*g      (mu != 0)
 *   d = g + mu*buf (Nesterov), buf (mu != 0), or g (mu = 0)
 *   p <- p - lr*d
 * with lr, wd, mu and 1 - dampening rounded from double to float once; then
 * the all-gather (or the owner's slice only, owner_only). The state's m is the
 * momentum buffer (a state without m serves only mu = 0); v is not used. The
 * parameter source is the owner's replica (fp32) or the master (mixed).
 * Algorithmic bytes per parameter: fp32 8N + 12 (8N + 4 without momentum),
 * mixed 4N + 16 (4N + 8 without momentum).
 * Errors: as zero_step_ex, plus EINVAL for a negative or non-finite momentum,
 * Nesterov without momentum or with dampening, or a state without m when
 * mu > 0. */
int zero_step_sgd(void *const *params, const void *const *grads, zero_states_t *st,
                  const zero_sgd_opts_t *opts, zero_stream_t stream);

/* ZeRO-3 gather(): all-gather the parameter shards into every replica
 * ("Data parallelism and ZeRO stages 1 to 3", section 2, stage 3, and
 * section 4, gather() before the forward pass). For every index j in
 * [lo, hi) with owner r (bounds[r] <= j < bounds[r+1], the state's shard
 * bounds), params[r][j] is copied into params[q][j] for every q != r; the
 * owner's element is only read. params: st->N device replicas of n elements
 * (float in ZERO_FP32, bf16 bits in ZERO_BF16_MIXED), disjoint; hi < 0 means
 * n. One kernel on `stream`, asynchronous; the copy is exact. Reads one and
 * writes N-1 elements per index.
 * Errors: EINVAL (NULL handle or replica, bad range, overlapping replicas),
 * EALIGN (a replica not aligned to its element size), ECUDA (launch). */
int zero_gather(void *const *params, zero_states_t *st, int64_t lo, int64_t hi,
                zero_stream_t stream);

/* --------------------------------------------------------------- buckets -- */

/* Gradient buckets ("ZeRO One: Sharding the Optimizer", section "Bucketing":
 * buckets of bucket_cap_mb * 1024 * 1024 bytes filled in backward order).
 * A bucket holds B = bucket_bytes / element_size consecutive elements of each
 * rank's gradient (element_size 4 for ZERO_FP32, 2 for ZERO_BF16_MIXED);
 * bucket k (k = 0 first ready) covers [max(0, n-(k+1)B), n-kB).
 * zero_bucket_count: *count = ceil(n / B). zero_bucket_range: bucket k's range.
 * Errors: EINVAL (n < 0, B < 1, bad precision, k outside [0, count), NULL). */
int zero_bucket_count(int64_t n, int32_t precision, int64_t bucket_bytes, int64_t *count);
int zero_bucket_range(int64_t n, int32_t precision, int64_t bucket_bytes, int64_t k,
                      int64_t *lo, int64_t *hi);

/* One bucket as soon as it is ready: queue on `side` a wait for `ready` (may
 * be NULL) and then the step on bucket k's range. `ready` must already have
 * been recorded by the producer when this is called (CUDA stream-wait
 * semantics). Errors: as zero_step_range, plus EINVAL for a bad k. */
int zero_step_bucket(void *const *params, const void *const *grads, zero_states_t *st,
                     int64_t t, double lr, double beta1, double beta2, double eps,
                     double weight_decay, int64_t bucket_bytes, int64_t k, zero_event_t ready,
                     zero_stream_t side);

/* The whole step, bucket by bucket, in arrival order: for k = 0..count-1 queue
 * on `side` a wait for ready[k] and the step on bucket k. `ready` holds
 * n_ready == count events (already recorded by the producer), or is NULL with
 * n_ready == 0 (no waits). `done` (may be NULL) is recorded on `side` after
 * the last bucket. With timeout_ms >= 0 the call then waits on the host, up
 * to timeout_ms milliseconds, for `done` (or for `side` when done is NULL)
 * and returns ZERO_ETIMEDOUT if the work is still running; the queued work
 * is not cancelled and completes later. With timeout_ms < 0 it returns after
 * queueing. The result equals zero_step bit for bit.
 * Errors: as zero_step, EINVAL for a bad bucket size or event count,
 * ETIMEDOUT. */
int zero_step_bucketed(void *const *params, const void *const *grads, zero_states_t *st,
                       int64_t t, double lr, double beta1, double beta2, double eps,
                       double weight_decay, int64_t bucket_bytes, const zero_event_t *ready,
                       int64_t n_ready, zero_stream_t side, zero_event_t done,
                       int64_t timeout_ms);

/* ------------------------------------------------------------ host input -- */

/* The step with the gradients in HOST memory, pipelined chunk by chunk. For
 * every chunk [lo, hi) of B = chunk_bytes / element_size elements, in index
 * order, this queues:
 *   on `h2d`     the copies host_grads[r][lo:hi] -> staging[r][lo:hi], all r;
 *   on `compute` the step on [lo, hi), once that chunk has arrived;
 *   on `d2h`     (host_params_out not NULL) the copy of the updated
 *                params[0][lo:hi] -> host_params_out[lo:hi].
 * Copies in both directions overlap the step of other chunks. The copies start
 * after everything already queued on `compute`; but when the step launches on
 * this handle since the previous call of this function were only that call's
 * own, with the same chunk size and staging buffers, the copy of chunk k waits
 * only for that call's step on chunk k, so back-to-back calls overlap. (The
 * staging buffers belong to these calls: nothing else may use them between
 * two such calls except through a step on this handle.) `compute` completes
 * only after the last chunk reached host_params_out, so synchronizing
 * `compute` covers the whole call.
 *   host_grads      : N HOST buffers of n elements, read-only (pinned memory
 *                     for asynchronous copies).
 *   staging         : N DEVICE buffers of n elements; they receive the
 *                     gradients and are the step's gradient buffers.
 *   host_params_out : NULL, or a HOST buffer of n elements.
 *   h2d, d2h        : streams for the two copy directions (streams distinct
 *                     from `compute` give the overlap; any streams are correct).
 * The result equals zero_step on the same gradients bit for bit. The handle
 * keeps 2*ceil(n/B)+2 CUDA events for these calls, created on first use;
 * calls on one handle must not run concurrently from several host threads.
 * Errors: as zero_step, plus EINVAL for a NULL host or staging buffer or a
 * chunk smaller than one element, ECUDA for a failed copy. */
int zero_step_from_host(void *const *params, const void *const *host_grads,
                        void *const *staging, zero_states_t *st, int64_t t, double lr,
                        double beta1, double beta2, double eps, double weight_decay,
                        void *host_params_out, int64_t chunk_bytes, zero_stream_t compute,
                        zero_stream_t h2d, zero_stream_t d2h);

/* zero_step_from_host with the options of zero_step_ex (AdamW) or of
 * zero_step_sgd (momentum SGD): exactly one of `adamw` and `sgd` is non-NULL.
 * Their step number, hyperparameters, grad_scale, clipping and owner_only are
 * used; the range must be the whole vector (lo = 0, hi = -1 or n).
 * Clipping (max_grad_norm > 0) needs norm_scratch (see zero_step_opts_t) and
 * norm_sq, an OUTPUT here: the global norm needs the whole gradient, so the
 * partial sums of each chunk's part of the norm run as soon as that chunk has
 * arrived, the fixed-order total once every chunk is in (bit for bit what
 * zero_grad_norm_sq gives on the staging buffers), and only then are the
 * chunks stepped in order, each copied back while the next is stepped.
 * With owner_only (ZeRO stage 3) the replicas stay released, and
 * host_params_out still receives the full updated parameters: each piece of a
 * chunk is copied from its owner's replica. Otherwise as zero_step_from_host.
 * SGD needs a state initialised for it (zero_init_states with v = NULL).
 * Errors: as zero_step_from_host, plus EINVAL for no or both option sets, a
 * partial range, bad options, clipping without norm_sq or norm_scratch, a
 * norm_scratch that is too small or overlaps a staging buffer; EALIGN for a
 * misaligned norm_sq or norm_scratch. */
int zero_step_from_host_ex(void *const *params, const void *const *host_grads,
                           void *const *staging, zero_states_t *st,
                           const zero_step_opts_t *adamw, const zero_sgd_opts_t *sgd,
                           void *host_params_out, int64_t chunk_bytes, zero_stream_t compute,
                           zero_stream_t h2d, zero_stream_t d2h);

/* ------------------------------------------------------------------- DDP -- */

/* DDP all_reduce(op="mean") in place ("Data parallelism and ZeRO stages 1 to 3",
 * section 2, "DDP": every rank gets the averaged gradient with identical
 * bits): grads[r][j] = (((g_0[j] + g_1[j]) + ...) + g_{N-1}[j]) / N for every
 * r, summed in fp32 in rank order; bf16 buffers receive the RNE of the fp32
 * mean. precision: ZERO_FP32 (float) or ZERO_BF16_MIXED (bf16).
 * Errors: EINVAL (n < 0, N outside [1, ZERO_MAX_RANKS], NULL, bad precision),
 * EALIGN, ECUDA. */
int ddp_allreduce_mean(void *const *grads, int64_t n, int32_t N, int32_t precision,
                       zero_stream_t stream);

/* ddp_allreduce_mean with the gradients in HOST memory, pipelined chunk by
 * chunk like zero_step_from_host. For every chunk [lo, hi) of B = chunk_bytes /
 * element_size elements, in index order, this queues:
 *   on `h2d`     the copies host_grads[r][lo:hi] -> staging[r][lo:hi], all r;
 *   on `compute` the mean of that chunk in place in the staging buffers, once
 *                it has arrived;
 *   on `d2h`     (host_mean_out not NULL) the copy of the mean
 *                staging[0][lo:hi] -> host_mean_out[lo:hi].
 * The copies start after everything already queued on `compute`, and
 * `compute` completes only after the last copy in either direction, so
 * synchronizing `compute` covers the whole call.
 *   host_grads    : N HOST buffers of n elements, read-only (pinned memory for
 *                   asynchronous copies).
 *   staging       : N DEVICE buffers of n elements, distinct and with the same
 *                   alignment rules as ddp_allreduce_mean; each ends holding
 *                   the mean, identical on every rank.
 *   host_mean_out : NULL, or a HOST buffer of n elements.
 * The staging buffers end bit for bit as ddp_allreduce_mean leaves device
 * buffers holding the same gradients. The library keeps a pool of CUDA events
 * per device for these calls (ceil(n/B)+2 at most), created on first use.
 * Errors: as ddp_allreduce_mean, plus EINVAL for a NULL host or staging
 * buffer or a chunk smaller than one element, ECUDA for a failed copy. */
int ddp_allreduce_mean_from_host(const void *const *host_grads, void *const *staging, int64_t n,
                                 int32_t N, int32_t precision, void *host_mean_out,
                                 int64_t chunk_bytes, zero_stream_t compute, zero_stream_t h2d,
                                 zero_stream_t d2h);

/* A host handle for back-to-back DDP means of host gradients. Consecutive
 * ddp_allreduce_mean_from_host_h calls on one handle with the same staging
 * buffers, n, N, precision and chunk size are chained chunk by chunk: the copy
 * of chunk k waits only for the previous call's mean of chunk k and its copy
 * back to the host, not for everything queued on `compute`, so the next call's
 * copies overlap the previous call's tail (the pipeline of "Data parallelism
 * and ZeRO stages 1 to 3", section 2, "DDP", over a stream of steps). The
 * staging buffers then belong to the handle's calls: device work that reads
 * or writes them between two calls (using the mean on the device, say) is not
 * waited for by the next call's copies unless the caller orders it on `h2d`,
 * or calls zero_ddp_host_reset first (the next call then waits for
 * everything queued on `compute`, as ddp_allreduce_mean_from_host always
 * does). A handle serves one device and one host thread at a time; it keeps
 * 2*ceil(n/B)+2 CUDA events, created on first use.
 * Errors: EINVAL (NULL), ENOMEM. */
typedef struct zero_ddp_host zero_ddp_host_t;
int zero_ddp_host_create(zero_ddp_host_t **out);
int zero_ddp_host_reset(zero_ddp_host_t *h);
int zero_ddp_host_free(zero_ddp_host_t *h); /* NULL is a no-op */

/* ddp_allreduce_mean_from_host on a handle (chained as described above); the
 * results are the same bits. Errors: as ddp_allreduce_mean_from_host, plus
 * EINVAL for a NULL handle or a handle used before on another device. */
int ddp_allreduce_mean_from_host_h(zero_ddp_host_t *h, const void *const *host_grads,
                                   void *const *staging, int64_t n, int32_t N, int32_t precision,
                                   void *host_mean_out, int64_t chunk_bytes, zero_stream_t compute,
                                   zero_stream_t h2d, zero_stream_t d2h);

/* ---------------------------------------------------------------- memory -- */

/* Model-state bytes per rank after a step, by stage: 0 = plain DDP, 1 = shard
 * the optimizer state, 2 = also the gradients, 3 = also the parameters
 * ("Data Parallelism & ZeRO", "ZeRO, stage by stage"; "Data parallelism and
 * ZeRO optimization", ZeRO-1/2/3 memory formulas). With per-parameter bytes
 * (P, G, K) = (4, 4, 8) for ZERO_FP32 and (2, 2, 12) for ZERO_BF16_MIXED, and
 * s the rank's shard size: params = P*(stage 3 ? s : n), grads =
 * G*(stage >= 2 ? s : n), optimizer = K*(stage >= 1 ? s : n). ZERO_FP64_EMU
 * reproduces the float64 bookkeeping table of "Data parallelism and ZeRO stages
 * 1 to 3", section 3 (stage 1 keeps the full averaged gradient plus the
 * chunk's; stages 1-2 hold m, v and a master chunk; stage 3 holds m, v).
 * zero_memory_breakdown writes {params, grads, optimizer} for `rank`;
 * zero_memory_bytes writes the total of rank 0, which holds the largest shard
 * (16n, 4n+12n/N, 2n+14n/N, 16n/N in mixed precision when N divides n).
 * Errors: EINVAL (n < 0, N < 1, stage outside 0..3, bad precision or rank,
 * NULL output, or a total that overflows 64 bits). */
int zero_memory_bytes(int64_t n, int32_t N, int32_t stage, int32_t precision, uint64_t *out);
int zero_memory_breakdown(int64_t n, int32_t N, int32_t stage, int32_t precision,
                          int32_t rank, uint64_t out[3]);
/* zero_memory_breakdown for caller-chosen shard bounds (HOST, N+1 offsets from
 * 0 to n; NULL: the np.array_split shards), e.g. whole-tensor shards. */
int zero_memory_breakdown_ex(int64_t n, int32_t N, int32_t stage, int32_t precision,
                             int32_t rank, const int64_t *bounds, uint64_t out[3]);

/* ---------------------------------------------------------------- errors -- */

/* Static description of a status code (never NULL). */
const char *zero_strerror(int code);
/* The calling thread's most recent error message ("" if none). */
const char *zero_last_error(void);

/* Failure injection for tests of the callers' error paths: the next `count`
 * handle allocations made by the calling thread (zero_init_states,
 * zero_init_states_ex, zero_ddp_host_create) fail with ZERO_ENOMEM, as if the
 * host allocator had returned NULL; nothing is queued and *out stays NULL.
 * count <= 0 clears a pending injection. Other threads are unaffected.
 * Returns ZERO_OK. */
int zero_debug_fail_host_allocs(int32_t count);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_H */
