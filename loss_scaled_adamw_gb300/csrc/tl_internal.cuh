// tl_internal.cuh - types shared by the kernels (tl_kernels.cu) and the host
// C ABI (tl_api.cu) of the GB300 loss-scaled AdamW library.  Not installed;
// the public interface is include/tl.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tl {

// Work decomposition (multi-tensor apply).  A segment is a piece of one tensor
// (at most kChunk elements), so it has one base pointer per list.  A chunk is
// either one segment of a large tensor, worked by a whole CTA, or a group of up
// to kGroup small tensors (at most kSmall elements each), one per warp.  The
// whole-CTA chunks come first in the table, then the groups, each part ordered
// by work, largest first, so that every round of a persistent grid (CTA b takes
// chunks b, b + G, b + 2G, ...) is balanced; the two parts run as separate
// launches.  Every run of chunks (a fixed piece of the table) writes its own
// squared-norm partials, so the reduction order (and the norm) does not depend on
// the grid size.
constexpr int kChunk = 16384;
#ifndef TL_SMALL
#define TL_SMALL 1024
#endif
constexpr int kSmall = TL_SMALL;
constexpr int kGroup = 8;            // = warps per CTA
#ifndef TL_RUN
#define TL_RUN 4
#endif
constexpr int kRun = TL_RUN;         // chunks per run where chunks are short (see launch_unscale)
constexpr int kThreads = 256;        // streaming kernels: 8 warps per CTA
// Threads per segment in the split forms (lists of short segments), where a CTA
// works several segments at once: 64 measured faster than 128 on the ragged
// 100k list (check pass 0.271 -> 0.259 ms, 0.380 -> 0.358 ms with gapped lists).
#ifndef TL_SPLIT_THREADS
#define TL_SPLIT_THREADS 64
#endif
constexpr int kSplitThreads = TL_SPLIT_THREADS;
static_assert(kSplitThreads % 32 == 0 && kSplitThreads > 32 && kThreads % kSplitThreads == 0,
              "a split form works a segment with whole warps (32 is the small-tensor form)");
constexpr int kNormThreads = 256;    // threads per CTA of the second-stage reduce
constexpr int kNormBlocks = 128;     // CTAs of the second-stage reduce: fixed, so its order is device-independent
constexpr int kInlineGrads = 512;    // gradient pointer tables up to this size travel in the kernel parameters

// Element types (values of TL_F32 / TL_BF16 / TL_F16 in include/tl.h).
constexpr int kF32 = 0;
constexpr int kBF16 = 1;
constexpr int kF16 = 2;
constexpr int kE4M3 = 3;   // 8-bit codes + fp32 scale per block of 16 (gradients only)
constexpr int kGradTypes = 4;

// One segment: elements [start, start + len) of tensor `tensor` (64 bytes).  The
// state-list addresses of its first element are stored in the descriptor, so a
// kernel reaches the data one load after the descriptor; the gradient lists,
// which change from call to call, are indexed by tensor and offset by start.
// gscale is the byte offset from a tensor's gradient pointer to its block
// scales (8-bit gradients: the codes rounded up to 16 bytes).
// In the whole-CTA part of the table chunk c is segment c; the groups that follow
// hold kGroup segments each (short groups padded with empty segments).
struct Chunk {
    float* acc;
    float* master;
    float* m;
    float* v;
    void* param;
    int64_t start;
    int32_t tensor;
    int32_t len;
    int64_t gscale;
};

// Device-resident scalars of one context.
struct DevState {
    float S;              // loss scale
    int32_t count;        // good steps since the last overflow or growth
    int64_t t;            // committed optimizer steps
    double b1p, b2p;      // beta1^t, beta2^t
    int32_t found_inf;    // overflow flag of the update in flight
    int32_t skipped;      // 1 if the last finished update was skipped
    float norm;           // global L2 norm of the unscaled gradient
    float coef;           // clip coefficient
    double sumsq;         // squared norm (fp64)
    uint32_t norm_ticket; // CTAs of the second-stage reduce that have finished, modulo 2^32
    uint32_t pass_ticket; // CTAs of a partial-writing launch that finish the norm in its last CTA (reset by it)
    uint32_t adam_ticket; // CTAs of the AdamW launch that runs the scaler in its last CTA (reset by it)
    int32_t run_slots;    // 1: one squared-norm slot per run (contexts that finish the norm in the pass),
                          // 0: one per warp per run (the 128-CTA second stage reads them)
};

// Gradient pointers passed by value (kernel parameter space).
struct GradTable {
    const void* p[kInlineGrads];
};

// Resident micro-batches read by one launch of the many-list kernel.
constexpr int kMaxMany = 8;
constexpr int kFewLists = 2;      // launches of at most this many lists use a kernel form of their own
constexpr int kRematLists = 4;    // lists an update may re-materialise u from (beyond, the resident pass moves fewer bytes)
constexpr int kInlineMany = 2048;  // k * ntensors gradient pointers travel by value up to this size

struct GradTableMany {
    const void* p[kInlineMany];     // list-major: p[i * ntensors + tensor]
};

struct ManyArgs {
    const void* const* tabs[kMaxMany];  // device pointer tables per list (nullptr: use the by-value table)
    float w[kMaxMany];                  // micro-batch weights n_i / N
    int32_t k;                          // micro-batches in this launch (1..kMaxMany)
    int32_t ntensors;
};

struct ScalerParams {
    int32_t enabled;
    float growth;
    float backoff;
    int32_t interval;
    float min_scale;
    float max_scale;
    int32_t run;     // 1: this launch runs the scaler state machine in its last CTA
};

struct AdamHP {
    float lr, beta1, beta2, eps, wd;
    float max_norm;         // the clip threshold of the update (<= 0: no clip)
    const float* lr_sched;  // device schedule: lr = lr_sched[min(t, lr_len - 1)] when set
    int64_t lr_len;
};

// Partial-writing launches of a context with at most this many chunks finish the
// norm in their last CTA (no separate reduce launch), and their runs write one
// squared-norm slot each (the warps' sums added by the CTA at the end of the run:
// fewer slots for the last CTA to read, for a block barrier per run); longer tables
// write one slot per warp per run, which the 128-CTA second stage reads, so that
// their warps never wait for each other at the end of a chunk.
#ifndef TL_FUSE_NORM_SLOTS
#define TL_FUSE_NORM_SLOTS 8192
#endif
constexpr int64_t kFuseNormSlots = TL_FUSE_NORM_SLOTS;

// What the a3 kernel reads besides the accumulation buffer.
enum UnscaleMode : int {
    kAccOnly = 0,   // u = acc / S
    kFirstOnly = 1, // u = (w * g) / S: the only micro-batch
    kAccAndGrad = 2 // u = fma(w, g, acc) / S: the last of several micro-batches
};

// Launchers (tl_kernels.cu).  Each streaming launcher covers chunks [c0, c1); the
// ones that write squared-norm partials take the chunks in runs of `run` (slots of
// the run's first chunk c: c, or c * kGroup + warp; see DevState::run_slots):
// small = false for whole-CTA chunks (one segment of a large tensor each),
// small = true for groups of small tensors (one warp per tensor).  `grid` is
// the persistent grid size; a gtab of nullptr means the pointers are in `inl`.
cudaError_t launch_accumulate(int gdt, bool first, bool small, const Chunk* chunks, int64_t c0,
                              int64_t c1, const GradTable& inl, const void* const* gtab, float w,
                              int grid, cudaStream_t s);
// fin > 0: this launch is the last of its pass and its last CTA reduces the fin
// partial slots of the whole table into the norm (sumsq, norm, overflow on a
// non-finite sum); fin = 0: a separate launch_norm does that.
cudaError_t launch_unscale(int gdt, int mode, bool small, const Chunk* chunks, int64_t c0,
                           int64_t c1, int run, const GradTable& inl, const void* const* gtab, float w,
                           DevState* st, double* partials, int64_t fin, int grid, cudaStream_t s);
// rot: the lists' element phases differ in some tensor (the rotated form, for the
// one- and two-list launches of 16-bit lists over whole-CTA segments).
cudaError_t launch_accum_many(int gdt, bool first, bool last, bool small, bool rot, const Chunk* chunks,
                              int64_t c0, int64_t c1, int run, const GradTableMany& inl,
                              const ManyArgs& a, DevState* st, double* partials, int64_t fin, int grid,
                              cudaStream_t s);
// The many-list pass without the store of u (all lists of the update at once),
// and the AdamW pass that recomputes u from the same lists.
cudaError_t launch_check_many(int gdt, bool small, bool rot, const Chunk* chunks, int64_t c0, int64_t c1, int run,
                              const GradTableMany& inl, const ManyArgs& a, DevState* st, double* partials,
                              int64_t fin, int grid, cudaStream_t s);
// The AdamW launches compute the clip coefficient from the device norm and
// hp.max_norm; with sp.run = 1 the launch's last CTA also runs the scaler state
// machine (the last AdamW launch of an update).  run: the part's run length (a
// whole-CTA launch with runs of several chunks takes the split form).
cudaError_t launch_adamw_remat(int pdt, int gdt, bool small, int run, const Chunk* chunks, int64_t c0,
                               int64_t c1, DevState* st, AdamHP hp, ScalerParams sp, const GradTableMany& inl,
                               const ManyArgs& a, int grid, cudaStream_t s);
cudaError_t launch_norm(const double* partials, int64_t n, double* slots, DevState* st, float max_norm,
                        cudaStream_t s);
cudaError_t launch_adamw(int pdt, bool small, int run, const Chunk* chunks, int64_t c0, int64_t c1,
                         DevState* st, AdamHP hp, ScalerParams sp, int grid, cudaStream_t s);
cudaError_t launch_seed(const DevState* st, float w, float* out, cudaStream_t s);
// One thread each: the clip coefficient from the device norm; the local squared norm
// and overflow flag copied out to caller memory; a global squared norm and flag
// (combined across shards by the caller) taken in as the update's norm.
cudaError_t launch_coef(DevState* st, float max_norm, cudaStream_t s);
cudaError_t launch_export(const DevState* st, double* sumsq, int32_t* flag, cudaStream_t s);
cudaError_t launch_import(DevState* st, const double* sumsq, const int32_t* flag, float max_norm, cudaStream_t s);

// The split forms of the streaming passes (tl_kernels_split.cu): each CTA works
// kThreads / kSplitThreads chunks at once.  launch_unscale, launch_accum_many,
// launch_check_many, launch_adamw and launch_adamw_remat hand them their whole-CTA
// launches of contexts with runs of several chunks (lists of short segments).
cudaError_t launch_unscale_split(int gdt, int mode, const Chunk* chunks, int64_t c0, int64_t c1, int run,
                                const GradTable& inl, const void* const* gtab, float w, DevState* st, double* partials,
                                int64_t fin, int grid, cudaStream_t s);
cudaError_t launch_accum_many_split(int gdt, bool first, bool last, bool rot, const Chunk* chunks, int64_t c0,
                                   int64_t c1, int run, const GradTableMany& inl, const ManyArgs& a, DevState* st,
                                   double* partials, int64_t fin, int grid, cudaStream_t s);
cudaError_t launch_check_many_split(int gdt, bool rot, const Chunk* chunks, int64_t c0, int64_t c1, int run,
                                   const GradTableMany& inl, const ManyArgs& a, DevState* st, double* partials,
                                   int64_t fin, int grid, cudaStream_t s);
cudaError_t launch_adamw_split(int pdt, const Chunk* chunks, int64_t c0, int64_t c1, DevState* st, AdamHP hp,
                               ScalerParams sp, int grid, cudaStream_t s);
cudaError_t launch_adamw_remat_split(int pdt, int gdt, const Chunk* chunks, int64_t c0, int64_t c1, DevState* st,
                                     AdamHP hp, ScalerParams sp, const GradTableMany& inl, const ManyArgs& a, int grid,
                                     cudaStream_t s);
int blocks_per_sm_split(int kind, int dt, int variant);

// Resident CTAs per SM of each streaming kernel (for persistent grid sizing).
// kind: 0 accumulate, 1 unscale, 2 adamw, 3 many-list accumulate (variant bit 0
// FIRST, bit 1 LAST, bit 2 at most kFewLists lists, bit 3 the rotated form), 4
// many-list pass without the store (variant bits 2, 3 as for kind 3), 5
// re-materialising adamw (dt = param dtype,
// variant bits 0-1 = grad dtype, bit 2 at most kFewLists lists).  For kinds 1, 3
// and 4, variant bit 4 asks for the form that a whole-CTA launch with runs of
// several chunks takes (the split form); kinds 2 and 5 likewise.
int blocks_per_sm(int kind, int dt, int variant, bool small);

}  // namespace tl
