/*
 * tl.h - C ABI of the GB300 loss-scaled AdamW optimizer step.
 *
 * One attempted logical update over k micro-batches is the call sequence
 *
 *     tl_accumulate(first=1) ; tl_accumulate(first=0) x (k-2) ;
 *     tl_unscale_check ; tl_grad_norm ; tl_clip_adamw_step ; tl_scaler_update
 *
 * (with k = 1: tl_unscale_check alone takes the only micro-batch), in the
 * order the Megatron page fixes ("Megatron Internals III: Mixed Precision,
 * Loss Scaling, and Grad Clipping", section 9 "The order matters": detect
 * overflow, copy gradients to fp32 main buffers, unscale, global norm, clip,
 * step fp32 masters, copy back).  Every call is asynchronous on the stream it
 * is given and never waits for the device, except tl_read_status,
 * tl_get_state and tl_set_state, which synchronise that stream.  The skip
 * decision, the loss scale and the optimizer step count live on the device:
 * no call reads a device value back to decide anything, so the whole
 * sequence can be enqueued (or captured) without a host synchronisation.
 *
 * Memory ownership.  The caller owns every tensor: the 16-bit model
 * parameters, the micro-batch gradients and the fp32 master weights, first
 * and second moments and accumulation buffer.  Pointers are device pointers
 * (or any address the device can load and store).  The library owns only
 * the opaque context: its chunk table, per-chunk norm partials, a cache of
 * gradient-pointer tables, and the device scalars (loss scale, good-step
 * count, optimizer step, beta powers, overflow flag, norm, clip coefficient).
 *
 * Tensor lists.  A tensor list is an array of ntensors pointers, tensor i
 * holding numel[i] contiguous elements.  Every list given to one context
 * uses the same ntensors and numel[].  Distinct tensors must not overlap,
 * in any list (a tensor passed twice would be counted twice in the global
 * norm; the tied input/output table appears once).  A pointer must be
 * aligned to its element size (8-bit gradient tensors: to 16 bytes).  A
 * segment whose streams are all 16-byte aligned, or all share their element
 * offset modulo 8 (tensors packed back to back in flat buffers), takes the
 * vector path after at most 7 scalar elements; streams of unequal offsets take
 * a scalar path (correct, slower).
 *
 * Errors.  Every function returns a status code; nothing is thrown across
 * this boundary.  A call that returns TL_EINVAL or TL_ESTATE has launched no
 * kernel and touched no caller memory (at most it has refreshed the context's
 * own cache of gradient pointer tables).  TL_ECUDA reports a failed CUDA call;
 * if a kernel launch of an update failed, part of that update may have run (the
 * overflow flag or the accumulation buffer half-written), so the context
 * abandons it and refuses every update call with TL_ESTATE until tl_set_state
 * has rewritten its scalars (from a tl_get_state snapshot, say).
 * Non-finite gradients are NOT an error: they set the device overflow flag
 * and the update is skipped on the device.
 *
 * Concurrency.  A context is not thread-safe: calls on one context must not
 * overlap in time (distinct contexts are independent).  The calls of one
 * update run in the order of the streams they are given; with more than one
 * stream the caller orders them (events), since each call reads what the
 * previous one wrote on the device.
 *
 * Pages cited (by title):
 *   [MP]  "Mixed precision, loss scaling, gradient accumulation, and
 *         activation checkpointing" (tinyllm module L11.1)
 *   [MEG] "Megatron Internals III: Mixed Precision, Loss Scaling, and Grad
 *         Clipping"
 *   [ZRO] "Your weights fit on one device but Adam's moments do not - how do
 *         you shard the optimizer state?"
 *   [RST] "Practical LLM in Rust", chapter 13 "Accumulate gradients and
 *         recompute activations"
 */
#ifndef TL_H
#define TL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define TL_OK 0
#define TL_EINVAL 1   /* bad argument: count, size, dtype, pointer, overlap, scaler setting */
#define TL_ECUDA 2    /* a CUDA runtime call or kernel launch failed */
#define TL_ESTATE 3   /* call out of order in the update sequence, or not allowed now */
#define TL_ENOMEM 4   /* the context could not allocate its own device/host memory */

/* Element types. */
#define TL_F32 0
#define TL_BF16 1
#define TL_F16 2
/* 8-bit gradients with fine-grained scaling ("Training at Scale", section 41.5:
 * one scale per block of values, the values stored in E4M3 relative to it and
 * dequantized before accumulation).  A gradient tensor of numel elements is one
 * buffer that starts on a 16-byte boundary: numel E4M3 codes (OCP layout: 1
 * sign, 4 exponent bits with bias 7, 3 mantissa bits; S.1111.111 is NaN),
 * padded to a multiple of 16 bytes, then ceil(numel / 16) fp32 block scales.
 * Element j of the tensor is the product, rounded to fp32, of the value of code
 * j and scale j / 16 (integer division); a tensor's last block may hold fewer
 * than 16 elements.  Gradient dtype only. */
#define TL_E4M3B16 3

typedef struct tl_ctx tl_ctx;

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef void* tl_stream;

/* Static configuration, fixed at tl_create.
 * [MP] section 4 "The interface": DynamicLossScaler(init=2^16, growth=2,
 * backoff=0.5, interval=2000); [MEG] section 5: the controller and its
 * min_loss_scale floor.  All five scale values must be powers of two so that
 * unscaling only changes exponents ([MP] section 2 "Loss scaling"), and the
 * loss scales at least 2^-126 (normal numbers, so that 1/S is finite).  With
 * scaler_enabled = 0 (bf16 training, [MP] "Dynamic scaling": bf16 needs no
 * scaler) S stays 1, the good-step count stays 0, and the finite check still
 * gates every update. */
typedef struct {
    int32_t param_dtype;    /* TL_BF16 or TL_F16: the model copy */
    int32_t grad_dtype;     /* TL_BF16, TL_F16, TL_F32 or TL_E4M3B16: the micro-batch gradients */
    int32_t scaler_enabled; /* 1: dynamic loss scaling; 0: S = 1 fixed */
    float init_scale;       /* S0 > 0, a power of two (e.g. 65536) */
    float growth;           /* > 1, a power of two (2) */
    float backoff;          /* in (0,1), a power of two (0.5) */
    int32_t interval;       /* >= 1 good steps between growths (2000) */
    float min_scale;        /* > 0, a power of two; S never goes below it (1) */
    float max_scale;        /* >= min_scale, a power of two; S never exceeds it (2^127) */
} tl_config;

/* AdamW hyper-parameters of one update (may change between updates, e.g.
 * under a learning-rate schedule).  beta1, beta2 in [0.5, 1), eps > 0,
 * lr >= 0, weight_decay >= 0. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} tl_adamw_hp;

/* The resumable scaler/optimizer scalars ([MP] section 4: state_dict keeps S
 * and the count; [RST] ch. 13: the optimizer state includes the beta powers
 * and the step).  b1p = beta1^t and b2p = beta2^t as products of the betas
 * actually used. */
typedef struct {
    float S;
    int32_t count;
    int64_t t;
    double b1p, b2p;
} tl_state;

/* Diagnostic snapshot (tests and logging). */
typedef struct {
    float S;            /* current loss scale */
    int32_t count;      /* good steps since the last overflow or growth */
    int64_t t;          /* committed optimizer steps */
    int32_t skipped;    /* 1 if the last finished update was skipped */
    int32_t found_inf;  /* overflow flag of the update in flight (0 once its AdamW launch has run) */
    float norm;         /* global L2 norm of the last update's unscaled gradient */
    float coef;         /* clip coefficient applied by the last update (<= 1) */
    double sumsq;       /* squared norm in fp64 */
    double b1p, b2p;
} tl_status;

/* Create a context for one tensor list.
 * ntensors >= 0; numel[i] >= 0.  param[i]: ntensors 16-bit model tensors of
 * param_dtype; master/m/v/acc[i]: fp32 tensors of the same sizes ([MEG]
 * section 1: fp16/bf16 param, fp32 master, fp32 Adam m and v; [MEG] section
 * 8: the fp32 master-gradient buffer).  The caller initialises master,
 * param, m and v; acc needs no initialisation.  Host arrays are copied
 * before return.  The context's device scalars start at S = init_scale
 * (1 when disabled), count 0, t 0, b1p = b2p = 1.  stream orders the
 * initial uploads; tl_create returns after they are complete.
 * Errors: TL_EINVAL (NULL/misaligned/overlapping pointers, bad sizes or
 * configuration), TL_ENOMEM, TL_ECUDA. */
int tl_create(tl_ctx** out, int64_t ntensors, const int64_t* numel, void* const* param,
              float* const* master, float* const* m, float* const* v, float* const* acc,
              const tl_config* cfg, tl_stream stream);

/* Release the context (waits for the device first).  NULL is accepted. */
int tl_destroy(tl_ctx* ctx);

/* Accumulate micro-batch i into the fp32 buffer (step a2).
 * [RST] ch. 13 "Weight each mean by the targets it represents": N = sum n_i,
 * the gradient of the mean over N targets is sum_i (n_i/N) grad L_i; [MP]
 * section 2 "Gradient accumulation": no zeroing in between.
 * grads: ntensors device pointers of grad_dtype, the gradient of micro-batch
 * i's MEAN loss times S.  n_i > 0 valid targets of this micro-batch, N the
 * total of the logical update (N <= 2^53, same N for every call of one
 * update).  w_i = fl32(n_i / N) computed in fp64 on the host.
 * first = 1: acc = w_i * g (starts an update, discarding any partial one);
 * first = 0: acc = fma(w_i, g, acc).
 * Errors: TL_EINVAL (counts, NULL pointer), TL_ESTATE (first = 0 with no
 * update open, or after tl_unscale_check). */
int tl_accumulate(tl_ctx* ctx, const void* const* grads, int64_t n_i, int64_t N, int first,
                  tl_stream stream);

/* Last micro-batch + unscale + overflow check + squared-norm partials (a3).
 * [MEG] section 8: cast, divide by the loss scale, place in the flattened
 * master-gradient buffer; [MEG] section 6: the overflow flag; [MP] "Loss
 * scaling": S a power of two makes unscaling exact.
 * u = (fma(w_k, g_k, acc), or w_k * g_k if no micro-batch was accumulated
 * before) * (1/S), stored into acc; the device overflow flag is raised if any
 * u is not finite; fp64 partial sums of fl32(u*u) are written (one per warp
 * of every chunk of the context's chunk table).
 * grads = NULL: all micro-batches were accumulated already (n_k ignored),
 * u = acc * (1/S).  The n_i of the update must total N by this call.
 * Errors: TL_EINVAL (counts do not add up to N), TL_ESTATE (out of order). */
int tl_unscale_check(tl_ctx* ctx, const void* const* grads, int64_t n_k, int64_t N,
                     tl_stream stream);

/* Several resident micro-batches in one pass (a2 for each, and a3 when last = 1).
 * For callers that keep the k micro-batch gradients resident (HBM is large on
 * this part): grads holds k lists of ntensors device pointers, list-major
 * (grads[i*ntensors + t] is tensor t of micro-batch i), n[i] their valid target
 * counts, N the total of the update.  Per element the result is bit-identical
 * to tl_accumulate(first=1) / tl_accumulate(first=0) ... / tl_unscale_check in
 * the same order: acc = w_1 g_1, acc = fma(w_i, g_i, acc), then with last = 1
 * u = acc * (1/S), the overflow flag and the squared-norm partials.  The fp32
 * buffer is written once per 8 micro-batches instead of once per micro-batch
 * (with k = 8: 2k + 4 bytes per parameter instead of 10k - 4).  Starts an
 * update when none is open, else continues it; with last = 1 the counts of the
 * update must total N, and the next call is tl_grad_norm.
 * Errors: TL_EINVAL (counts, NULL pointers), TL_ESTATE (out of order). */
int tl_accumulate_many(tl_ctx* ctx, int k, const void* const* grads, const int64_t* n, int64_t N, int last,
                       tl_stream stream);

/* A whole logical update over k <= 4 resident micro-batches without storing u
 * (a2 for each and a3, re-materialising form).  [MEG] section 8 (real
 * implementations fuse and flatten the copy / unscale / check path).  Reads the
 * k lists (same layout as tl_accumulate_many) once and computes, per element and
 * in registers only, u = fma(w_k, g_k, ... fma(w_2, g_2, w_1 g_1)) * (1/S): the
 * operations and order of tl_accumulate_many, so the same u bit for bit.  It
 * raises the overflow flag and writes the squared-norm partials; acc is neither
 * read nor written.  tl_grad_norm follows as usual, and tl_clip_adamw_step then
 * recomputes u from the same k lists instead of reading it from acc.  HBM bytes
 * per parameter for the update: 26 + 4k (16-bit grads) instead of the resident
 * pass's 34 + 2k, fewer for k < 4.  Opens an update (none may be open) and
 * covers all of it: the counts must total N.  The context keeps the k lists'
 * pointers (not their data) until tl_clip_adamw_step has been enqueued; the
 * gradients must stay unchanged in device memory until that step has run.
 * Errors: TL_EINVAL (k outside 1..4, counts, NULL or overlapping pointers),
 * TL_ESTATE (an update is open). */
int tl_unscale_check_many(tl_ctx* ctx, int k, const void* const* grads, const int64_t* n, int64_t N,
                          tl_stream stream);

/* Global L2 norm and clip coefficient (a4).  [MEG] section 9: global_norm =
 * sqrt(sum ||grad||^2), clip_coef = max_norm / (global_norm + eps); the
 * coefficient is applied only when below 1 (eps = 1e-6); max_norm <= 0
 * disables clipping (coef = 1, the norm is still computed).  The partials
 * are reduced in a fixed order, so the norm is deterministic.  A non-finite
 * squared norm raises the overflow flag.  Where the device work happens: for
 * a context of at most 8,192 chunks the pass of tl_unscale_check (or of the
 * last tl_accumulate_many, or tl_unscale_check_many) reduces the norm in its
 * last CTA and this call launches nothing; longer tables get a second-stage
 * launch here.  Either way the AdamW launch derives the coefficient from the
 * device norm and this max_norm.  Errors: TL_ESTATE. */
int tl_grad_norm(tl_ctx* ctx, float max_norm, tl_stream stream);

/* The sharded form of a4, for an update whose tensor list is split over
 * several contexts (one per rank of a sharded optimizer, each owning a slice of
 * the parameters, see tl_partition).  "Megatron Internals III", section 6
 * "Overflow must be global": all ranks of one logical update take the same
 * step-or-skip decision (the flag is all-reduced with max); section 9 and
 * [ZRO] "Operational sharp edges", "Gradient clipping": each rank sums the
 * squares of its own slice, those scalars are all-reduced (sum) before the
 * square root is taken, and every rank clips with the same coefficient.
 * tl_local_sumsq (in place of tl_grad_norm, after the pass) writes this
 * context's squared norm (fp64) and overflow flag (0 or 1) into caller device
 * memory on the stream, without any host synchronisation.  The caller
 * combines them across ranks (e.g. an all-reduce: sum of the squared norms,
 * max of the flags) into device memory, and tl_grad_norm_from takes the
 * combined values as the update's: sumsq, norm = sqrt(sumsq), the flag raised
 * if the combined flag is set or the sum is not finite, and the clip
 * coefficient from max_norm.  tl_clip_adamw_step and tl_scaler_update follow
 * as usual, so every rank skips or steps together and moves S identically.
 *   d_sumsq: one double, 8-byte aligned; d_flag: one int32, 4-byte aligned
 *   (device memory, owned by the caller).
 * Errors: TL_EINVAL (pointers, max_norm NaN), TL_ESTATE (out of order). */
int tl_local_sumsq(tl_ctx* ctx, double* d_sumsq, int32_t* d_flag, tl_stream stream);
int tl_grad_norm_from(tl_ctx* ctx, const double* d_sumsq, const int32_t* d_flag, float max_norm,
                      tl_stream stream);

/* The slice of a tensor list that rank `rank` of nranks owns in a sharded
 * optimizer ([ZRO] "The scheme": partition the parameter vector into N
 * disjoint slices, slice i on device i; "Partition granularity": slicing the
 * flat vector splits tensors across owners).  The list is flattened in tensor
 * order, then element order (P elements); the cuts are b_j = the largest
 * multiple of align not above floor(j * P / nranks) for j = 0 .. nranks - 1,
 * and b_nranks = P.  Rank r owns [b_r, b_(r+1)), returned as pieces in tensor
 * order: piece q is elements [start[q], start[q] + len[q]) of tensor
 * tensor[q]; empty pieces are left out, so *count <= ntensors.  A context over
 * a rank's pieces takes each state tensor's address plus start (and the same
 * for the gradients).  align (>= 1) keeps the cuts on multiples of align
 * elements (16 keeps 8-bit gradient blocks whole inside a tensor that starts
 * on a block).  Host only: no CUDA call.  *count is always written; the pieces
 * are written only when cap >= *count.
 * Errors: TL_EINVAL (sizes, nranks < 1, rank outside [0, nranks), align < 1,
 * cap too small, NULL arrays). */
int tl_partition(int64_t ntensors, const int64_t* numel, int32_t nranks, int32_t rank, int64_t align,
                 int64_t* tensor, int64_t* start, int64_t* len, int64_t cap, int64_t* count);

/* How tl_create lays out a tensor list, from its sizes alone (host only: no
 * CUDA call).  The list becomes a table of chunks: whole-CTA segments (pieces
 * of at most `seg` elements of one tensor; seg is the longest power of two from
 * 16,384 down to 4,096 that still gives at least 24 segments per SM) and, when
 * the list holds at least 128 tensors of at most 1,024 elements, groups of up
 * to 8 such tensors worked one per warp.  Runs of chunks write the squared-norm
 * partials: one chunk per run where the segments are mostly full, 4 where they
 * are short, and then the passes take the split forms (several segments per
 * CTA).  A table of at most 8,192 chunks finishes the norm in the last CTA of
 * the partial-writing pass (tl_grad_norm then launches nothing).
 * sm_count: the SM count of the device the context will run on (152 on a
 * GB300; tl_create reads it from the device).  The environment variable
 * TL_SMALL_GROUP_MIN, when set, replaces the 128 (as it does for tl_create).
 * Errors: TL_EINVAL (ntensors < 0, NULL arrays, a negative size, sm_count < 1,
 * a list too large to index). */
typedef struct {
    int64_t nchunks;     /* chunks of the table: nbig + ngroups */
    int64_t nbig;        /* whole-CTA segments */
    int64_t ngroups;     /* groups of up to 8 small tensors */
    int64_t seg;         /* segment length, elements */
    int64_t nsmall;      /* tensors in the groups */
    int32_t run_big;     /* chunks per squared-norm run, whole-CTA part (1 or 4) */
    int32_t run_small;   /* ... in the groups (4) */
    int32_t split_forms; /* 1: the whole-CTA part takes the split forms */
    int32_t fused_norm;  /* 1: the partial-writing pass finishes the norm */
} tl_plan_info;

int tl_plan(int64_t ntensors, const int64_t* numel, int32_t sm_count, tl_plan_info* out);

/* Clip + AdamW on the fp32 masters + recast to the model dtype (a5).
 * [MEG] sections 7 and 9 (clip with the global coefficient, step the fp32
 * masters, copy back to model precision); [ZRO] "Why the optimizer state is
 * the thing that overflows" (bias-corrected first moment over the root of
 * the bias-corrected second moment plus a small constant); [RST] ch. 13
 * (decoupled weight decay; beta powers as state).  Per element, in fp32 with
 * each operation rounded to nearest:
 *   g = u*coef; m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g);
 *   w = w - (lr*wd)*w; w = w - (lr/(1-b1^(t+1))) * (m / (sqrt(v)/sqrt(1-b2^(t+1)) + eps));
 *   param = round-to-nearest-even(w).
 * u is read from acc, or, after tl_unscale_check_many, recomputed from the
 * micro-batch lists that call was given.
 * If the overflow flag is set the kernel exits without touching any tensor.
 * Errors: TL_EINVAL (hp), TL_ESTATE. */
int tl_clip_adamw_step(tl_ctx* ctx, const tl_adamw_hp* hp, tl_stream stream);

/* Learning-rate schedule read on the device.  With a schedule set, the update
 * that would commit optimizer step t+1 (t = committed steps, the device count)
 * takes lr = lr_table[min(t, len-1)] in place of hp->lr; the other
 * hyper-parameters still come from tl_clip_adamw_step.  The index counts
 * committed steps only, so an update skipped on overflow leaves the next
 * scheduled rate for the next attempt ([RST] ch. 13 "Discard a failed partial
 * logical update": the optimizer step stays and the scheduled step remains
 * available; "Carry one logical update into schedule reasoning": warm-up and
 * decay are per logical update).  Because the rate is chosen on the device, a
 * skipped step needs no host read, and a captured CUDA graph follows the
 * schedule on every replay.
 *   lr_table: len fp32 rates (entry i for optimizer step i+1) in memory the
 *     device can read (device, managed or pinned host), 4-byte aligned; owned
 *     by the caller, who keeps it alive and its values finite and >= 0 while
 *     it is set.  It is read when each AdamW kernel runs, so entries may be
 *     rewritten between updates in stream order.
 *   len = 0 (lr_table ignored) removes the schedule: hp->lr applies again.
 * Takes effect for the tl_clip_adamw_step calls made after it (a CUDA graph
 * keeps the table address it was captured with).  Host-only; launches nothing.
 * Errors: TL_EINVAL (len < 0; lr_table NULL, misaligned or not readable by
 * the device when len > 0). */
int tl_set_lr_schedule(tl_ctx* ctx, const float* lr_table, int64_t len);

/* Scaler state machine and optimizer scalars (a6).  [MEG] section 5; [MP]
 * "Dynamic scaling" and the five-step trace of section 3; [RST] ch. 13
 * "Discard a failed partial logical update".
 * Overflow: S = max(S*backoff, min_scale), count = 0, t and the beta powers
 * unchanged, skipped = 1.  Clean: t += 1, beta powers advanced, count += 1,
 * and when count reaches interval S = min(S*growth, max_scale), count = 0.
 * The overflow flag is cleared.  The device work runs in the last CTA of the
 * AdamW launch of tl_clip_adamw_step (after every CTA has read S and the
 * flag), so a status read after tl_clip_adamw_step already shows it; this
 * call closes the update on the host and launches nothing.
 * Errors: TL_ESTATE. */
int tl_scaler_update(tl_ctx* ctx, tl_stream stream);

/* Synchronous reads and writes of the device scalars (these wait for the
 * stream).  tl_read_status between tl_grad_norm and tl_clip_adamw_step first
 * computes the clip coefficient of the update in flight on the device.
 * tl_set_state is allowed only between updates and checks S
 * (power of two within [min_scale, max_scale], or 1 when disabled), count
 * (0 <= count < interval) and t >= 0 ([MP] section 4 catalogue: a resume
 * keeps S and the count; bad arguments raise).  Errors: TL_EINVAL,
 * TL_ESTATE, TL_ECUDA. */
int tl_read_status(tl_ctx* ctx, tl_status* out, tl_stream stream);
int tl_get_state(tl_ctx* ctx, tl_state* out, tl_stream stream);
int tl_set_state(tl_ctx* ctx, const tl_state* in, tl_stream stream);

/* Device address of the current loss scale S (fp32), for scaling the loss
 * on the device without a host read ([MP] section 4: scale(loss) = loss*S).
 * Valid until tl_destroy. */
const float* tl_scale_ptr(const tl_ctx* ctx);

/* The backward seed of micro-batch i: S * n_i / N in fp32, written by the device
 * to out (one float of device memory) at the point of the stream where it runs,
 * so the loss can be seeded without a host read of S ([RST] ch. 13 "Weight each
 * mean by the targets it represents": reverse mode is seeded with S * n_i / N;
 * [MP] section 4: scale(loss) = loss * S).  With S a power of two the value is
 * exactly S * fl32(n_i / N).  Errors: TL_EINVAL (counts, out NULL). */
int tl_loss_seed(tl_ctx* ctx, int64_t n_i, int64_t N, float* out, tl_stream stream);

/* Sizes of the context: total elements and work chunks. */
int64_t tl_num_params(const tl_ctx* ctx);
int64_t tl_num_chunks(const tl_ctx* ctx);

/* Result of tl_unscale_norm_noalloc, written by the device into caller memory. */
typedef struct {
    float norm;         /* global L2 norm of the unscaled gradient */
    float coef;         /* clip coefficient (<= 1; 1 when max_norm <= 0) */
    int32_t found_inf;  /* 1 if some unscaled element, or the squared norm, is not finite */
    int32_t reserved;
    double sumsq;       /* squared norm in fp64 */
} tl_norm_result;

/* Unscale + overflow check + global norm + clip coefficient WITHOUT ANY
 * ALLOCATION.  No passage of the pages has a counterpart: this entry point
 * exists for callers that cannot call cudaMalloc (device memory owned by
 * another allocator, no allocation allowed after start-up, or an allocation
 * that would disturb a capture or a memory plan), who therefore cannot use
 * tl_create.  It needs no context.
 * acc: ntensors fp32 device tensors of numel[i] elements (4-byte aligned),
 * holding the accumulated scaled gradient; they are overwritten with
 * u = acc * (1/S).  S: a power of two, at least 2^-126 (so that 1/S is exact
 * and finite).  max_norm <= 0 disables clipping.  out: device memory (8-byte
 * aligned) that receives the result.  u and the overflow rule are those of
 * tl_unscale_check (u bit for bit); the squared norm is summed in another
 * order (fp32 over 8 squares, fp64 beyond), so norm and sumsq agree with
 * tl_grad_norm to 1e-6 relative, not bit for bit.
 * Scratch: a fixed array inside the library, 512 KiB of fp64 partials, held
 * by every GPU that loads it until the process exits.  Under CUDA's lazy
 * module loading (the default) the array is created on a device by the FIRST
 * call of this function there, which therefore takes device memory once and
 * can fail for want of it; later calls allocate nothing.  Make that first
 * call on each device before any stream capture and before handing all
 * device memory to another allocator (or set CUDA_MODULE_LOADING=EAGER).
 * Limits: ntensors <= 256 and at most 2^16 chunks of 16,384 elements (2^30
 * elements); larger lists give TL_EINVAL.  Every call shares the scratch and
 * writes every partial it reads; calls that overlap on the GPU race on it.
 * Errors: TL_EINVAL (sizes, pointers, S), TL_ECUDA. */
int tl_unscale_norm_noalloc(int64_t ntensors, const int64_t* numel, float* const* acc, float S,
                            float max_norm, tl_norm_result* out, tl_stream stream);

/* Number of kernels this context has launched so far. */
int64_t tl_launch_count(const tl_ctx* ctx);

/* Human-readable text of a status code, and of the last error a context saw. */
const char* tl_status_string(int status);
const char* tl_last_error(const tl_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* TL_H */
