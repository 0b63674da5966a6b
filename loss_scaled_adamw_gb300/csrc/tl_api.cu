// tl_api.cu - host side of the C ABI declared in include/tl.h.
//
// Holds the opaque context: argument validation (all of it before any work is
// enqueued), the chunk table of the multi-tensor-apply launcher (built once per
// tensor list and kept on the device), the norm partials, the device
// scalars, a cache of device-resident gradient pointer tables for lists too
// long to pass by value, and the order of the calls of one logical update.
#include "tl_internal.cuh"

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/tl.h"

using namespace tl;

namespace {

enum Phase { kIdle = 0, kAccum = 1, kUnscaled = 2, kNormed = 3, kStepped = 4, kLocal = 5 };

// Segment length: the longest power of two in [kMinSeg, kChunk] that still gives the
// whole-CTA part at least kSegPerSm segments per SM, so that a persistent grid of a
// few CTAs per SM gets several rounds of similar segments (a list of ~10M elements
// in 16,384-element segments would give barely two rounds, and its last round would
// run on a fraction of the grid).  Long lists keep kChunk.
#ifndef TL_SEG_MIN
#define TL_SEG_MIN 4096
#endif
#ifndef TL_SEG_PER_SM
#define TL_SEG_PER_SM 24
#endif
constexpr int64_t kMinSeg = TL_SEG_MIN;
constexpr int64_t kSegPerSm = TL_SEG_PER_SM;
// Small tensors are grouped one per warp (a part of the table with its own launch)
// only when the list holds at least this many of them; fewer small tensors become
// whole-CTA segments of their own, so the pass is one launch.  The environment
// variable TL_SMALL_GROUP_MIN (read by make_plan, for tl_create and tl_plan)
// overrides it (tests set 1 to run the group kernels on short lists).
constexpr int64_t kGroupMin = 128;

int elem_size(int dt) { return dt == TL_F32 ? 4 : dt == TL_E4M3B16 ? 1 : 2; }

// Bytes of one gradient tensor of n elements (8-bit: codes padded to 16 bytes,
// then one fp32 scale per block of 16).
uintptr_t grad_bytes(int dt, int64_t n) {
    if (dt == TL_E4M3B16) return uintptr_t((n + 15) / 16 * 16 + (n + 15) / 16 * 4);
    return uintptr_t(n) * uintptr_t(elem_size(dt));
}

// A normal power of two (>= 2^-126): unscaling by it only changes exponents and
// its reciprocal is finite.
bool is_pow2(float x) {
    if (!(x >= FLT_MIN) || !std::isfinite(x)) return false;
    int e = 0;
    return std::frexp(x, &e) == 0.5f;
}

struct Interval {
    uintptr_t lo, hi;  // [lo, hi)
};

// A device-resident gradient pointer table keyed by the host pointer array.
struct GradSlot {
    std::vector<const void*> key;
    uint64_t hash = 0;
    const void** d_tab = nullptr;   // ntensors device pointers
    const void** h_stage = nullptr; // pinned staging copy
    cudaEvent_t last_use = nullptr;
    uint64_t stamp = 0;
    bool valid = false;
};

constexpr int kGradSlots = 16;

uint64_t hash_ptrs(const void* const* p, int64_t n) {
    uint64_t h = 1469598103934665603ull;
    for (int64_t i = 0; i < n; ++i) {
        h ^= reinterpret_cast<uintptr_t>(p[i]);
        h *= 1099511628211ull;
    }
    return h;
}

}  // namespace

struct tl_ctx {
    int device = 0;
    int sm_count = 0;
    tl_config cfg{};
    int64_t ntensors = 0;
    int64_t P = 0;
    int64_t nchunks = 0;
    std::vector<int64_t> numel;
    std::vector<Interval> state_iv;  // sorted intervals of every state tensor
    Chunk* d_chunks = nullptr;     // segments
    double* d_partials = nullptr;
    double* d_norm_slots = nullptr;  // one per CTA of the second-stage reduce
    DevState* d_state = nullptr;
    GradSlot slots[kGradSlots];
    uint64_t clock = 0;
    int64_t nbig = 0;              // chunks [0, nbig) are whole-CTA segments, [nbig, nchunks) small-tensor groups
    int64_t seg = kChunk;          // segment length of this list (a power of two <= kChunk)
    // the partial-writing pass finishes the norm in its last CTA (few partial slots);
    // else tl_grad_norm launches the 128-CTA second stage
    bool fuse_norm = false;
    float max_norm = 0.0f;         // clip threshold of the update in flight (set by tl_grad_norm / _from)
    // persistent grid sizes per kernel variant, [..][0] for the whole-CTA part, [..][1] for the groups
    int grid_acc[kGradTypes][2][2] = {};
    int grid_uns[kGradTypes][3][2] = {};
    int grid_adam[3][2] = {};
    int grid_many[kGradTypes][16][2] = {};
    int grid_check[kGradTypes][2][2][2] = {};     // [grad dtype][few lists][rotated form][part]
    // the state lists hold tensors whose streams share no element phase (a gapped
    // layout): the one- and two-list many-list launches take their rotated form,
    // taking the gradient lists to follow the same kind of layout
    bool gapped = false;
    // chunks per run of the kernels that write norm partials, per part: 1 where the
    // chunks are mostly full segments, kRun where they are short (one warp
    // reduction per run instead of per chunk)
    int run[2] = {1, 1};
    int grid_remat[3][kGradTypes][2][2] = {};     // [param dtype][grad dtype][few lists][part]
    // the update in flight
    int phase = kIdle;
    int64_t n_sum = 0;
    int64_t N_update = 0;
    bool accumulated = false;
    // a failed launch interrupted an update: its kernels may have run in part (the
    // overflow flag or acc half-written), so no update runs until tl_set_state
    bool interrupted = false;
    // host-side fault injection for tests (environment TL_TEST_FAIL_LAUNCH=n at
    // tl_create): the context's n-th kernel launch reports a failure instead of
    // launching
    int64_t fail_at = 0;
    int64_t attempts = 0;
    // a re-materialising update: u was never stored; the step recomputes it from
    // these lists (list-major, ntensors pointers each) and counts
    bool remat = false;
    int remat_k = 0;
    std::vector<const void*> remat_grads;
    int64_t remat_n[kRematLists] = {};
    // learning-rate schedule read by the AdamW kernels (caller-owned; null: hp.lr)
    const float* lr_sched = nullptr;
    int64_t lr_len = 0;
    int64_t launches = 0;
    std::string last_error;
};

namespace {

int fail(tl_ctx* ctx, int code, const std::string& msg) {
    if (ctx != nullptr) ctx->last_error = msg;
    return code;
}

int cuda_fail(tl_ctx* ctx, cudaError_t e, const char* what) {
    std::string msg = std::string(what) + ": " + cudaGetErrorString(e);
    return fail(ctx, TL_ECUDA, msg);
}

// A launch of an update's kernels failed: the update is abandoned.
int launch_fail(tl_ctx* ctx, cudaError_t e, const char* what) {
    ctx->interrupted = true;
    ctx->phase = kIdle;  // tl_set_state may run
    return cuda_fail(ctx, e, what);
}

int refuse_if_interrupted(tl_ctx* ctx) {
    if (!ctx->interrupted) return TL_OK;
    return fail(ctx, TL_ESTATE, "a failed launch interrupted an update; restore the scalars with tl_set_state");
}

bool overlaps_any(const std::vector<Interval>& sorted, uintptr_t lo, uintptr_t hi) {
    // sorted by lo and pairwise disjoint: only the last interval starting before hi can overlap
    auto it = std::lower_bound(sorted.begin(), sorted.end(), hi,
                               [](const Interval& a, uintptr_t v) { return a.lo < v; });
    if (it == sorted.begin()) return false;
    --it;
    return it->hi > lo;
}

int check_config(const tl_config* c, std::string& why) {
    if (c->param_dtype != TL_BF16 && c->param_dtype != TL_F16) { why = "param_dtype must be TL_BF16 or TL_F16"; return TL_EINVAL; }
    if (c->grad_dtype != TL_BF16 && c->grad_dtype != TL_F16 && c->grad_dtype != TL_F32 && c->grad_dtype != TL_E4M3B16) { why = "grad_dtype must be TL_BF16, TL_F16, TL_F32 or TL_E4M3B16"; return TL_EINVAL; }
    if (c->scaler_enabled != 0 && c->scaler_enabled != 1) { why = "scaler_enabled must be 0 or 1"; return TL_EINVAL; }
    if (c->scaler_enabled) {
        if (!is_pow2(c->init_scale)) { why = "init_scale must be a positive power of two"; return TL_EINVAL; }
        if (!is_pow2(c->growth) || !(c->growth > 1.0f)) { why = "growth must be a power of two > 1"; return TL_EINVAL; }
        if (!is_pow2(c->backoff) || !(c->backoff < 1.0f)) { why = "backoff must be a power of two < 1"; return TL_EINVAL; }
        if (c->interval < 1) { why = "interval must be >= 1"; return TL_EINVAL; }
        if (!is_pow2(c->min_scale) || !is_pow2(c->max_scale) || c->min_scale > c->max_scale) {
            why = "min_scale and max_scale must be powers of two with min_scale <= max_scale"; return TL_EINVAL;
        }
        if (c->init_scale < c->min_scale || c->init_scale > c->max_scale) { why = "init_scale must lie in [min_scale, max_scale]"; return TL_EINVAL; }
    }
    return TL_OK;
}

int check_counts(tl_ctx* ctx, int64_t n_i, int64_t N) {
    if (N <= 0 || N > (int64_t(1) << 53)) return fail(ctx, TL_EINVAL, "N must be in [1, 2^53]");
    if (n_i <= 0 || n_i > N) return fail(ctx, TL_EINVAL, "n_i must be in [1, N]");
    return TL_OK;
}

int check_device(tl_ctx* ctx) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDevice");
    if (dev != ctx->device) return fail(ctx, TL_ESTATE, "the current CUDA device is not the context's device");
    return TL_OK;
}

// Validate a gradient list against the context (sizes implied, alignment, no
// overlap with anything the kernels write).
int check_grads(tl_ctx* ctx, const void* const* grads) {
    const int dt = ctx->cfg.grad_dtype;
    // 8-bit gradients: each tensor's codes start on a 16-byte boundary, so its
    // segments (multiples of 16 elements apart) never split an 8-element vector
    // across two scale blocks
    const uintptr_t align = dt == TL_E4M3B16 ? 16 : uintptr_t(elem_size(dt));
    for (int64_t i = 0; i < ctx->ntensors; ++i) {
        if (ctx->numel[i] == 0) continue;
        const uintptr_t a = reinterpret_cast<uintptr_t>(grads[i]);
        if (a == 0) return fail(ctx, TL_EINVAL, "NULL gradient pointer for tensor " + std::to_string(i));
        if (a % align != 0) return fail(ctx, TL_EINVAL, "misaligned gradient pointer for tensor " + std::to_string(i));
        if (overlaps_any(ctx->state_iv, a, a + grad_bytes(dt, ctx->numel[i])))
            return fail(ctx, TL_EINVAL, "gradient tensor " + std::to_string(i) + " overlaps a state tensor");
    }
    return TL_OK;
}

// Resolve the gradient table for one call: by value when short, else a cached
// device table (uploaded on first use of this exact pointer list).
int resolve_device_table(tl_ctx* ctx, const void* const* grads, cudaStream_t s, const void* const** dtab,
                         GradSlot** used);

int resolve_grads(tl_ctx* ctx, const void* const* grads, cudaStream_t s, GradTable* inl,
                  const void* const** dtab, GradSlot** used) {
    *dtab = nullptr;
    *used = nullptr;
    if (ctx->ntensors <= kInlineGrads) {
        int rc = check_grads(ctx, grads);
        if (rc != TL_OK) return rc;
        for (int64_t i = 0; i < ctx->ntensors; ++i) inl->p[i] = grads[i];
        return TL_OK;
    }
    return resolve_device_table(ctx, grads, s, dtab, used);
}

// A device-resident copy of one gradient pointer list, from the cache (uploaded
// on the first use of this exact list).
int resolve_device_table(tl_ctx* ctx, const void* const* grads, cudaStream_t s, const void* const** dtab,
                         GradSlot** used) {
    *dtab = nullptr;
    *used = nullptr;
    const uint64_t h = hash_ptrs(grads, ctx->ntensors);
    ctx->clock += 1;
    for (GradSlot& sl : ctx->slots) {
        if (sl.valid && sl.hash == h && std::equal(sl.key.begin(), sl.key.end(), grads)) {
            sl.stamp = ctx->clock;
            *dtab = sl.d_tab;
            *used = &sl;
            return TL_OK;
        }
    }
    int rc = check_grads(ctx, grads);
    if (rc != TL_OK) return rc;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
        return fail(ctx, TL_ESTATE, "a new gradient list cannot be uploaded during stream capture; use it once before capturing");
    GradSlot* victim = &ctx->slots[0];
    for (GradSlot& sl : ctx->slots) {
        if (!sl.valid) { victim = &sl; break; }
        if (sl.stamp < victim->stamp) victim = &sl;
    }
    if (victim->valid && victim->last_use != nullptr) {
        cudaError_t e = cudaEventSynchronize(victim->last_use);  // its previous users are done
        if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventSynchronize");
    }
    std::memcpy(victim->h_stage, grads, sizeof(void*) * size_t(ctx->ntensors));
    cudaError_t e = cudaMemcpyAsync(victim->d_tab, victim->h_stage, sizeof(void*) * size_t(ctx->ntensors),
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemcpyAsync(gradient table)");
    victim->key.assign(grads, grads + ctx->ntensors);
    victim->hash = h;
    victim->stamp = ctx->clock;
    victim->valid = true;
    *dtab = victim->d_tab;
    *used = victim;
    return TL_OK;
}

void mark_used(GradSlot* sl, cudaStream_t s) {
    if (sl == nullptr || sl->last_use == nullptr) return;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone)
        cudaEventRecord(sl->last_use, s);
}

int grid_for(tl_ctx* ctx, int per_sm, int64_t nchunks) {
    int64_t g = int64_t(ctx->sm_count) * per_sm;
    if (g > nchunks) g = nchunks;
    if (g < 1) g = 1;
    return int(g);
}

// Every kernel launch of an update passes here first (the test fault injection).
cudaError_t gate(tl_ctx* ctx) {
    ctx->attempts += 1;
    return ctx->fail_at > 0 && ctx->attempts == ctx->fail_at ? cudaErrorLaunchFailure : cudaSuccess;
}

// Launch one streaming operation over the chunk table: the whole-CTA part and
// the small-tensor groups are separate launches (launch(small, c0, c1, last), last
// true for the final launch of the operation).
template <typename Launch>
cudaError_t over_parts(tl_ctx* ctx, Launch launch) {
    const bool groups = ctx->nchunks > ctx->nbig;
    if (ctx->nbig > 0) {
        cudaError_t e = gate(ctx);
        if (e == cudaSuccess) e = launch(false, int64_t(0), ctx->nbig, !groups);
        if (e != cudaSuccess) return e;
        ctx->launches += 1;
    }
    if (groups) {
        cudaError_t e = gate(ctx);
        if (e == cudaSuccess) e = launch(true, ctx->nbig, ctx->nchunks, true);
        if (e != cudaSuccess) return e;
        ctx->launches += 1;
    }
    return cudaSuccess;
}

// Partial slots the last launch of a partial-writing pass reduces itself (0: the
// norm is left to the second-stage launch of tl_grad_norm).
int64_t fin_slots(const tl_ctx* ctx, bool last) {
    return ctx->fuse_norm && last ? ctx->nchunks : 0;   // one slot per run (DevState::run_slots)
}

// Resolve (and validate) k gradient lists (list-major, ntensors pointers each)
// before any launch: a table by value when k lists fit in it, else one cached
// device table per list.
int resolve_lists(tl_ctx* ctx, int k, const void* const* grads, cudaStream_t s, bool* by_value,
                  std::vector<const void* const*>& tabs, std::vector<GradSlot*>& slots) {
    const int64_t nt = ctx->ntensors;
    *by_value = nt <= kInlineMany / kMaxMany;
    tabs.assign(size_t(k), nullptr);
    slots.assign(size_t(k), nullptr);
    if (nt == 0) return TL_OK;
    for (int i = 0; i < k; ++i) {
        const void* const* gi = grads + int64_t(i) * nt;
        int rc = *by_value ? check_grads(ctx, gi) : resolve_device_table(ctx, gi, s, &tabs[size_t(i)], &slots[size_t(i)]);
        if (rc != TL_OK) return rc;
    }
    return TL_OK;
}

// The kernel arguments of lists [j, j + kk) of a resolved set.
void fill_many_args(const tl_ctx* ctx, const void* const* grads, const int64_t* n, int64_t N, int j, int kk,
                    bool by_value, const std::vector<const void* const*>& tabs, ManyArgs& a, GradTableMany& inl) {
    const int64_t nt = ctx->ntensors;
    a = ManyArgs{};
    a.k = kk;
    a.ntensors = static_cast<int32_t>(nt);
    for (int i = 0; i < kk; ++i) {
        a.w[i] = static_cast<float>(static_cast<double>(n[j + i]) / static_cast<double>(N));
        a.tabs[i] = by_value ? nullptr : tabs[size_t(j + i)];
        if (by_value)
            for (int64_t t = 0; t < nt; ++t) inl.p[int64_t(i) * nt + t] = grads[int64_t(j + i) * nt + t];
    }
}

void free_ctx(tl_ctx* ctx) {
    if (ctx == nullptr) return;
    cudaFree(ctx->d_chunks);
    cudaFree(ctx->d_partials);
    cudaFree(ctx->d_norm_slots);
    cudaFree(ctx->d_state);
    for (GradSlot& sl : ctx->slots) {
        cudaFree(sl.d_tab);
        cudaFreeHost(sl.h_stage);
        if (sl.last_use != nullptr) cudaEventDestroy(sl.last_use);
    }
    delete ctx;
}

// The chunk table of a tensor list, decided from the sizes and the SM count alone
// (tl_create adds each segment's state addresses; tl_plan reports it).  A large
// tensor becomes one segment per `seg` elements; small tensors (<= kSmall elements)
// are grouped kGroup to a chunk, one per warp, when there are at least
// small_group_min() of them.  Chunks are then ordered by work, largest first
// (stable): the whole-CTA part, then the groups, so every round of a persistent
// grid gets chunks of similar size.
struct PlanSeg {
    int64_t tensor, start, len;
};
struct PlanChunk {
    std::vector<PlanSeg> segs;
    int64_t work = 0;
    bool group = false;
};
struct Plan {
    int64_t seg = kChunk;           // segment length
    std::vector<PlanChunk> chunks;  // whole-CTA chunks, then the groups
    int64_t nbig = 0;               // whole-CTA chunks
    int run[2] = {1, 1};            // chunks per squared-norm run, per part (whole-CTA, groups)
    bool fuse_norm = false;         // the partial-writing pass finishes the norm (one slot per run)
};

int64_t small_group_min() {
    if (const char* g = std::getenv("TL_SMALL_GROUP_MIN")) return std::max<int64_t>(1, std::atoll(g));
    return kGroupMin;
}

// numel: ntensors sizes, validated by the caller (non-negative, P within range).
Plan make_plan(int64_t ntensors, const int64_t* numel, int sm_count) {
    Plan pl;
    int64_t P = 0, n_small = 0, small_elems = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        if (numel[i] <= 0) continue;
        P += numel[i];
        if (numel[i] <= kSmall) { ++n_small; small_elems += numel[i]; }
    }
    const bool grouping = n_small >= small_group_min();
    const int64_t whole = P - (grouping ? small_elems : 0);
    int64_t seg = kChunk;
    while (seg > kMinSeg && whole / seg < kSegPerSm * sm_count) seg /= 2;
    pl.seg = seg;
    PlanChunk group;
    group.group = true;
    for (int64_t i = 0; i < ntensors; ++i) {
        if (numel[i] <= 0) continue;
        if (grouping && numel[i] <= kSmall) {
            group.segs.push_back(PlanSeg{i, 0, numel[i]});
            group.work += numel[i];
            if (int(group.segs.size()) == kGroup) {
                pl.chunks.push_back(std::move(group));
                group = PlanChunk();
                group.group = true;
            }
            continue;
        }
        for (int64_t st = 0; st < numel[i]; st += seg) {
            PlanChunk one;
            const int64_t len = std::min<int64_t>(seg, numel[i] - st);
            one.segs.push_back(PlanSeg{i, st, len});
            one.work = len;
            pl.chunks.push_back(std::move(one));
        }
    }
    if (!group.segs.empty()) pl.chunks.push_back(std::move(group));
    std::stable_sort(pl.chunks.begin(), pl.chunks.end(), [](const PlanChunk& a, const PlanChunk& b) {
        if (a.group != b.group) return b.group;
        return a.work > b.work;
    });
    int64_t big_elems = 0;
    for (const PlanChunk& cb : pl.chunks) {
        if (cb.group) continue;
        ++pl.nbig;
        big_elems += cb.work;
    }
    // chunks are mostly full segments: one squared-norm partial each; where they are
    // short (one warp or a few), kRun of them per partial, which also selects the split
    // forms of the partial-writing and AdamW passes
    pl.run[0] = pl.nbig > 0 && big_elems < pl.nbig * (seg / 2) ? kRun : 1;
    pl.run[1] = kRun;
    const int64_t nchunks = int64_t(pl.chunks.size());
    pl.fuse_norm = nchunks > 0 && nchunks <= kFuseNormSlots;
    return pl;
}

}  // namespace

extern "C" {

const char* tl_status_string(int status) {
    switch (status) {
        case TL_OK: return "ok";
        case TL_EINVAL: return "invalid argument";
        case TL_ECUDA: return "CUDA error";
        case TL_ESTATE: return "call not allowed in the current state";
        case TL_ENOMEM: return "out of memory";
        default: return "unknown status";
    }
}

const char* tl_last_error(const tl_ctx* ctx) {
    return ctx == nullptr ? "" : ctx->last_error.c_str();
}

int tl_create(tl_ctx** out, int64_t ntensors, const int64_t* numel, void* const* param, float* const* master,
              float* const* m, float* const* v, float* const* acc, const tl_config* cfg, tl_stream stream) {
    if (out == nullptr || cfg == nullptr) return TL_EINVAL;
    *out = nullptr;
    if (ntensors < 0 || ntensors > (int64_t(1) << 31) - 1) return TL_EINVAL;
    if (ntensors > 0 && (numel == nullptr || param == nullptr || master == nullptr || m == nullptr ||
                         v == nullptr || acc == nullptr))
        return TL_EINVAL;
    std::string why;
    if (check_config(cfg, why) != TL_OK) return TL_EINVAL;
    const int pes = elem_size(cfg->param_dtype);

    // Sizes, pointers, alignment and overlap: everything before any allocation.
    std::vector<Interval> iv;
    iv.reserve(size_t(ntensors) * 5);
    int64_t P = 0, nchunks = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        if (numel[i] < 0) return TL_EINVAL;
        if (numel[i] == 0) continue;
        if (numel[i] > (int64_t(1) << 62) / 4 - P) return TL_EINVAL;
        P += numel[i];
        nchunks += (numel[i] + kChunk - 1) / kChunk;
        const void* ptrs[5] = {param[i], master[i], m[i], v[i], acc[i]};
        for (int l = 0; l < 5; ++l) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(ptrs[l]);
            const int es = l == 0 ? pes : 4;
            if (a == 0 || a % es != 0) return TL_EINVAL;
            iv.push_back({a, a + uintptr_t(numel[i]) * es});
        }
    }
    // a gapped layout: some tensor's state streams are neither all on a 16-byte boundary
    // nor all at one element phase modulo 8
    bool gapped = false;
    for (int64_t i = 0; i < ntensors && !gapped; ++i) {
        if (numel[i] == 0) continue;
        const uintptr_t a[5] = {reinterpret_cast<uintptr_t>(param[i]), reinterpret_cast<uintptr_t>(master[i]),
                                reinterpret_cast<uintptr_t>(m[i]), reinterpret_cast<uintptr_t>(v[i]),
                                reinterpret_cast<uintptr_t>(acc[i])};
        bool al = true, same = true;
        const uintptr_t r0 = (a[1] / 4) & 7;
        for (int l = 0; l < 5; ++l) {
            al = al && (a[l] & 15u) == 0;
            same = same && ((a[l] / (l == 0 ? uintptr_t(pes) : 4)) & 7) == r0;
        }
        gapped = !al && !same;
    }
    std::sort(iv.begin(), iv.end(), [](const Interval& a, const Interval& b) { return a.lo < b.lo; });
    for (size_t k = 1; k < iv.size(); ++k)
        if (iv[k].lo < iv[k - 1].hi) return TL_EINVAL;  // two tensors share memory

    tl_ctx* ctx = new (std::nothrow) tl_ctx();
    if (ctx == nullptr) return TL_ENOMEM;
    ctx->cfg = *cfg;
    ctx->gapped = gapped;
    ctx->ntensors = ntensors;
    ctx->P = P;
    ctx->nchunks = nchunks;
    ctx->numel.assign(numel, numel + ntensors);
    ctx->state_iv = std::move(iv);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device);
    if (const char* f = std::getenv("TL_TEST_FAIL_LAUNCH")) ctx->fail_at = std::atoll(f);
    if (e != cudaSuccess) { free_ctx(ctx); return TL_ECUDA; }

    // The chunk table (make_plan), with each segment's state addresses.  Whole-CTA
    // chunk c is segment c; every group holds kGroup segments, a short group padded
    // with empty segments (its first tensor, length 0) so that a warp finds its
    // tensor without an index table.
    const Plan pl = make_plan(ntensors, numel, ctx->sm_count);
    ctx->seg = pl.seg;
    const int64_t nbig = pl.nbig;
    auto seg = [&](const PlanSeg& q) {
        const int64_t i = q.tensor, st = q.start;
        return Chunk{acc[i] + st, master[i] + st, m[i] + st, v[i] + st,
                     static_cast<char*>(param[i]) + st * pes, st, int32_t(i), int32_t(q.len), (numel[i] + 15) / 16 * 16};
    };
    std::vector<Chunk> chunks;
    chunks.reserve(size_t(nbig) + (pl.chunks.size() - size_t(nbig)) * kGroup);
    for (size_t b = 0; b < pl.chunks.size(); ++b) {
        const PlanChunk& cb = pl.chunks[b];
        for (const PlanSeg& q : cb.segs) chunks.push_back(seg(q));
        if (int64_t(b) >= nbig) {
            Chunk pad = seg(cb.segs[0]);
            pad.len = 0;
            for (size_t i = cb.segs.size(); i < size_t(kGroup); ++i) chunks.push_back(pad);
        }
    }
    nchunks = int64_t(pl.chunks.size());
    ctx->nchunks = nchunks;
    ctx->nbig = nbig;
    const size_t nc_alloc = size_t(std::max<int64_t>(nchunks, 1));
    if (cudaMalloc(&ctx->d_chunks, sizeof(Chunk) * std::max<size_t>(chunks.size(), 1)) != cudaSuccess ||
        cudaMalloc(&ctx->d_partials, sizeof(double) * nc_alloc * kGroup) != cudaSuccess ||
        cudaMalloc(&ctx->d_norm_slots, sizeof(double) * kNormBlocks) != cudaSuccess ||
        cudaMalloc(&ctx->d_state, sizeof(DevState)) != cudaSuccess) {
        cudaGetLastError();
        free_ctx(ctx);
        return TL_ENOMEM;
    }
    if (ntensors > kInlineMany / kMaxMany) {
        for (GradSlot& sl : ctx->slots) {
            if (cudaMalloc(reinterpret_cast<void**>(&sl.d_tab), sizeof(void*) * size_t(ntensors)) != cudaSuccess ||
                cudaMallocHost(reinterpret_cast<void**>(&sl.h_stage), sizeof(void*) * size_t(ntensors)) != cudaSuccess ||
                cudaEventCreateWithFlags(&sl.last_use, cudaEventDisableTiming) != cudaSuccess) {
                cudaGetLastError();
                free_ctx(ctx);
                return TL_ENOMEM;
            }
        }
    }
    DevState ds{};
    ds.S = cfg->scaler_enabled ? cfg->init_scale : 1.0f;
    ds.count = 0;
    ds.t = 0;
    ds.b1p = 1.0;
    ds.b2p = 1.0;
    ds.found_inf = 0;
    ds.skipped = 0;
    ds.norm = 0.0f;
    ds.coef = 1.0f;
    ds.sumsq = 0.0;
    ds.norm_ticket = 0;
    ds.pass_ticket = 0;
    ds.adam_ticket = 0;
    // contexts that finish the norm in the pass write one partial slot per run
    ctx->fuse_norm = pl.fuse_norm;
    ds.run_slots = ctx->fuse_norm ? 1 : 0;
    e = cudaMemcpyAsync(ctx->d_state, &ds, sizeof(ds), cudaMemcpyHostToDevice, s);
    // partial slots not at the start of a run stay zero for good
    if (e == cudaSuccess) e = cudaMemsetAsync(ctx->d_partials, 0, sizeof(double) * nc_alloc * kGroup, s);
    if (e == cudaSuccess && nchunks > 0)
        e = cudaMemcpyAsync(ctx->d_chunks, chunks.data(), sizeof(Chunk) * chunks.size(), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) { free_ctx(ctx); return TL_ECUDA; }

    // Persistent grid sizes from the occupancy of each kernel variant the
    // context's dtypes can launch.
    const int gdt = cfg->grad_dtype, pdt = cfg->param_dtype;
    ctx->run[0] = pl.run[0];
    ctx->run[1] = pl.run[1];
    for (int part = 0; part < 2; ++part) {
        const bool small = part == 1;
        const int64_t n = small ? nchunks - nbig : nbig;
        const int64_t nruns = (n + ctx->run[part] - 1) / ctx->run[part];
        // the partial-writing passes over runs of several chunks take their split form
        const int hf = !small && ctx->run[part] > 1 ? 16 : 0;
        for (int f = 0; f < 2; ++f) ctx->grid_acc[gdt][f][part] = grid_for(ctx, blocks_per_sm(0, gdt, f, small), n);
        for (int md = 0; md < 3; ++md)
            ctx->grid_uns[gdt][md][part] = grid_for(ctx, blocks_per_sm(1, gdt, md | hf, small), nruns);
        ctx->grid_adam[pdt][part] = grid_for(ctx, blocks_per_sm(2, pdt, hf, small), n);
        for (int vr = 0; vr < 16; ++vr)
            ctx->grid_many[gdt][vr][part] = grid_for(ctx, blocks_per_sm(3, gdt, vr | hf, small), nruns);
        for (int few = 0; few < 2; ++few) {
            for (int rt = 0; rt < 2; ++rt)
                ctx->grid_check[gdt][few][rt][part] =
                    grid_for(ctx, blocks_per_sm(4, gdt, (few ? 4 : 0) | (rt ? 8 : 0) | hf, small), nruns);
            ctx->grid_remat[pdt][gdt][few][part] =
                grid_for(ctx, blocks_per_sm(5, pdt, gdt | (few ? 4 : 0) | hf, small), n);
        }
    }
    *out = ctx;
    return TL_OK;
}

int tl_destroy(tl_ctx* ctx) {
    if (ctx == nullptr) return TL_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_ctx(ctx);
    return e == cudaSuccess ? TL_OK : TL_ECUDA;
}

int tl_accumulate(tl_ctx* ctx, const void* const* grads, int64_t n_i, int64_t N, int first, tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (grads == nullptr && ctx->ntensors > 0) return fail(ctx, TL_EINVAL, "grads must not be NULL");
    if (first != 0 && first != 1) return fail(ctx, TL_EINVAL, "first must be 0 or 1");
    int rc = check_counts(ctx, n_i, N);
    if (rc != TL_OK) return rc;
    if (first) {
        if (ctx->phase != kIdle && ctx->phase != kAccum)
            return fail(ctx, TL_ESTATE, "an update is past its accumulation phase; finish it with tl_scaler_update");
    } else {
        if (ctx->phase != kAccum) return fail(ctx, TL_ESTATE, "first=0 with no update open");
        if (N != ctx->N_update) return fail(ctx, TL_EINVAL, "N differs from the N of the open update");
        if (n_i > N - ctx->n_sum) return fail(ctx, TL_EINVAL, "the counts exceed N");
    }
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    static thread_local GradTable inl;
    const void* const* dtab = nullptr;
    GradSlot* used = nullptr;
    if (ctx->ntensors > 0 && (rc = resolve_grads(ctx, grads, s, &inl, &dtab, &used)) != TL_OK) return rc;
    const float w = static_cast<float>(static_cast<double>(n_i) / static_cast<double>(N));
    if (ctx->nchunks > 0) {
        const int gdt = ctx->cfg.grad_dtype;
        cudaError_t e = over_parts(ctx, [&](bool small, int64_t c0, int64_t c1, bool) {
            return launch_accumulate(gdt, first != 0, small, ctx->d_chunks, c0, c1, inl,
                                     dtab, w, ctx->grid_acc[gdt][first][small ? 1 : 0], s);
        });
        if (e != cudaSuccess) return launch_fail(ctx, e, "accumulate launch");
        mark_used(used, s);
    }
    if (first) {
        ctx->N_update = N;
        ctx->n_sum = 0;
    }
    ctx->n_sum += n_i;
    ctx->accumulated = true;
    ctx->phase = kAccum;
    return TL_OK;
}

int tl_unscale_check(tl_ctx* ctx, const void* const* grads, int64_t n_k, int64_t N, tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    int mode;
    int rc;
    if (grads == nullptr) {
        if (ctx->phase != kAccum) return fail(ctx, TL_ESTATE, "no accumulated micro-batch to unscale");
        if (ctx->n_sum != ctx->N_update) return fail(ctx, TL_EINVAL, "the accumulated counts do not add up to N");
        mode = kAccOnly;
    } else {
        if ((rc = check_counts(ctx, n_k, N)) != TL_OK) return rc;
        if (ctx->phase == kIdle) {
            if (n_k != N) return fail(ctx, TL_EINVAL, "the only micro-batch must have n_k == N");
            mode = kFirstOnly;
        } else if (ctx->phase == kAccum) {
            if (N != ctx->N_update) return fail(ctx, TL_EINVAL, "N differs from the N of the open update");
            if (ctx->n_sum + n_k != N) return fail(ctx, TL_EINVAL, "the counts do not add up to N");
            mode = kAccAndGrad;
        } else {
            return fail(ctx, TL_ESTATE, "tl_unscale_check called twice in one update");
        }
    }
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    static thread_local GradTable inl;
    const void* const* dtab = nullptr;
    GradSlot* used = nullptr;
    if (grads != nullptr && ctx->ntensors > 0 && (rc = resolve_grads(ctx, grads, s, &inl, &dtab, &used)) != TL_OK)
        return rc;
    const float w = grads == nullptr ? 1.0f : static_cast<float>(static_cast<double>(n_k) / static_cast<double>(N));
    if (ctx->nchunks > 0) {
        const int gdt = ctx->cfg.grad_dtype;
        cudaError_t e = over_parts(ctx, [&](bool small, int64_t c0, int64_t c1, bool lastl) {
            return launch_unscale(gdt, mode, small, ctx->d_chunks, c0, c1, ctx->run[small ? 1 : 0], inl, dtab, w,
                                  ctx->d_state, ctx->d_partials, fin_slots(ctx, lastl),
                                  ctx->grid_uns[gdt][mode][small ? 1 : 0], s);
        });
        if (e != cudaSuccess) return launch_fail(ctx, e, "unscale launch");
        mark_used(used, s);
    }
    if (grads != nullptr) {
        if (ctx->phase == kIdle) ctx->N_update = N;
        ctx->n_sum = ctx->phase == kIdle ? n_k : ctx->n_sum + n_k;
    }
    ctx->phase = kUnscaled;
    return TL_OK;
}

int tl_accumulate_many(tl_ctx* ctx, int k, const void* const* grads, const int64_t* n, int64_t N, int last,
                       tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (k < 1 || n == nullptr) return fail(ctx, TL_EINVAL, "need k >= 1 micro-batches and their counts");
    if (grads == nullptr && ctx->ntensors > 0) return fail(ctx, TL_EINVAL, "grads must not be NULL");
    if (last != 0 && last != 1) return fail(ctx, TL_EINVAL, "last must be 0 or 1");
    int rc;
    int64_t sum = 0;
    for (int i = 0; i < k; ++i) {
        if ((rc = check_counts(ctx, n[i], N)) != TL_OK) return rc;
        sum += n[i];
        if (sum > N) return fail(ctx, TL_EINVAL, "the counts exceed N");
    }
    bool first;
    if (ctx->phase == kIdle) {
        first = true;
    } else if (ctx->phase == kAccum) {
        first = false;
        if (N != ctx->N_update) return fail(ctx, TL_EINVAL, "N differs from the N of the open update");
        if (sum > N - ctx->n_sum) return fail(ctx, TL_EINVAL, "the counts exceed N");
    } else {
        return fail(ctx, TL_ESTATE, "an update is past its accumulation phase; finish it with tl_scaler_update");
    }
    const int64_t total = (first ? 0 : ctx->n_sum) + sum;
    if (last && total != N) return fail(ctx, TL_EINVAL, "the counts do not add up to N");
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    static thread_local GradTableMany inl;
    // Resolve (and validate) every list before the first launch, so that an
    // error leaves nothing enqueued.
    bool by_value = true;
    std::vector<const void* const*> tabs;
    std::vector<GradSlot*> slots;
    if ((rc = resolve_lists(ctx, k, grads, s, &by_value, tabs, slots)) != TL_OK) return rc;
    for (int j = 0; j < k; j += kMaxMany) {
        const int kk = std::min(kMaxMany, k - j);
        ManyArgs a;
        fill_many_args(ctx, grads, n, N, j, kk, by_value, tabs, a, inl);
        const bool f = first && j == 0;
        const bool l = last && j + kk == k;
        if (ctx->nchunks > 0) {
            const int vr = (f ? 1 : 0) | (l ? 2 : 0) | (kk <= kFewLists ? 4 : 0) | (ctx->gapped ? 8 : 0);
            const int gdt = ctx->cfg.grad_dtype;
            cudaError_t e = over_parts(ctx, [&](bool small, int64_t c0, int64_t c1, bool lastl) {
                return launch_accum_many(gdt, f, l, small, ctx->gapped, ctx->d_chunks, c0, c1, ctx->run[small ? 1 : 0], inl, a,
                                         ctx->d_state, ctx->d_partials, fin_slots(ctx, lastl),
                                         ctx->grid_many[gdt][vr][small ? 1 : 0], s);
            });
            if (e != cudaSuccess) return launch_fail(ctx, e, "many-list accumulate launch");
            for (int i = 0; i < kk; ++i) mark_used(slots[j + i], s);
        }
    }
    if (first) ctx->N_update = N;
    ctx->n_sum = total;
    ctx->accumulated = true;
    ctx->phase = last ? kUnscaled : kAccum;
    return TL_OK;
}

int tl_unscale_check_many(tl_ctx* ctx, int k, const void* const* grads, const int64_t* n, int64_t N,
                          tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (k < 1 || k > kRematLists || n == nullptr)
        return fail(ctx, TL_EINVAL, "need 1 <= k <= " + std::to_string(kRematLists) + " micro-batches and their counts");
    if (grads == nullptr && ctx->ntensors > 0) return fail(ctx, TL_EINVAL, "grads must not be NULL");
    if (ctx->phase != kIdle)
        return fail(ctx, TL_ESTATE, "tl_unscale_check_many opens an update: finish the open one with tl_scaler_update");
    int rc;
    int64_t sum = 0;
    for (int i = 0; i < k; ++i) {
        if ((rc = check_counts(ctx, n[i], N)) != TL_OK) return rc;
        sum += n[i];
        if (sum > N) return fail(ctx, TL_EINVAL, "the counts exceed N");
    }
    if (sum != N) return fail(ctx, TL_EINVAL, "the counts do not add up to N");
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    static thread_local GradTableMany inl;
    bool by_value = true;
    std::vector<const void* const*> tabs;
    std::vector<GradSlot*> slots;
    if ((rc = resolve_lists(ctx, k, grads, s, &by_value, tabs, slots)) != TL_OK) return rc;
    if (ctx->nchunks > 0) {
        ManyArgs a;
        fill_many_args(ctx, grads, n, N, 0, k, by_value, tabs, a, inl);
        const int gdt = ctx->cfg.grad_dtype;
        const int few = k <= kFewLists ? 1 : 0;
        cudaError_t e = over_parts(ctx, [&](bool small, int64_t c0, int64_t c1, bool lastl) {
            return launch_check_many(gdt, small, ctx->gapped, ctx->d_chunks, c0, c1, ctx->run[small ? 1 : 0], inl, a,
                                     ctx->d_state, ctx->d_partials, fin_slots(ctx, lastl),
                                     ctx->grid_check[gdt][few][ctx->gapped ? 1 : 0][small ? 1 : 0],
                                     s);
        });
        if (e != cudaSuccess) return launch_fail(ctx, e, "many-list check launch");
        for (int i = 0; i < k; ++i) mark_used(slots[size_t(i)], s);
    }
    ctx->remat = true;
    ctx->remat_k = k;
    ctx->remat_grads.assign(grads, grads + int64_t(k) * ctx->ntensors);
    for (int i = 0; i < k; ++i) ctx->remat_n[i] = n[i];
    ctx->N_update = N;
    ctx->n_sum = N;
    ctx->accumulated = true;
    ctx->phase = kUnscaled;
    return TL_OK;
}

int tl_grad_norm(tl_ctx* ctx, float max_norm, tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (ctx->phase != kUnscaled) return fail(ctx, TL_ESTATE, "tl_grad_norm must follow tl_unscale_check");
    if (std::isnan(max_norm)) return fail(ctx, TL_EINVAL, "max_norm is NaN");
    int rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    // With the norm finished by the pass itself there is nothing to launch: the AdamW
    // launch derives the clip coefficient from the device norm and max_norm.
    if (!ctx->fuse_norm) {
        cudaError_t e = gate(ctx);
        if (e == cudaSuccess)
            e = launch_norm(ctx->d_partials, ctx->nchunks * kGroup, ctx->d_norm_slots, ctx->d_state, max_norm,
                            static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return launch_fail(ctx, e, "norm launch");
        ctx->launches += 1;
    }
    ctx->max_norm = max_norm;
    ctx->phase = kNormed;
    return TL_OK;
}

int tl_local_sumsq(tl_ctx* ctx, double* d_sumsq, int32_t* d_flag, tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (ctx->phase != kUnscaled) return fail(ctx, TL_ESTATE, "tl_local_sumsq must follow tl_unscale_check");
    if (d_sumsq == nullptr || (reinterpret_cast<uintptr_t>(d_sumsq) & 7u) != 0 || d_flag == nullptr ||
        (reinterpret_cast<uintptr_t>(d_flag) & 3u) != 0)
        return fail(ctx, TL_EINVAL, "d_sumsq (8-byte aligned) and d_flag (4-byte aligned) must be device addresses");
    int rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (!ctx->fuse_norm) {
        e = gate(ctx);
        if (e == cudaSuccess) e = launch_norm(ctx->d_partials, ctx->nchunks * kGroup, ctx->d_norm_slots, ctx->d_state,
                                              0.0f, s);
        if (e != cudaSuccess) return launch_fail(ctx, e, "norm launch");
        ctx->launches += 1;
    }
    e = gate(ctx);
    if (e == cudaSuccess) e = launch_export(ctx->d_state, d_sumsq, d_flag, s);
    if (e != cudaSuccess) return launch_fail(ctx, e, "export launch");
    ctx->launches += 1;
    ctx->phase = kLocal;
    return TL_OK;
}

int tl_grad_norm_from(tl_ctx* ctx, const double* d_sumsq, const int32_t* d_flag, float max_norm, tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (ctx->phase != kLocal) return fail(ctx, TL_ESTATE, "tl_grad_norm_from must follow tl_local_sumsq");
    if (std::isnan(max_norm)) return fail(ctx, TL_EINVAL, "max_norm is NaN");
    if (d_sumsq == nullptr || (reinterpret_cast<uintptr_t>(d_sumsq) & 7u) != 0 || d_flag == nullptr ||
        (reinterpret_cast<uintptr_t>(d_flag) & 3u) != 0)
        return fail(ctx, TL_EINVAL, "d_sumsq (8-byte aligned) and d_flag (4-byte aligned) must be device addresses");
    int rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaError_t e = gate(ctx);
    if (e == cudaSuccess) e = launch_import(ctx->d_state, d_sumsq, d_flag, max_norm, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return launch_fail(ctx, e, "import launch");
    ctx->launches += 1;
    ctx->max_norm = max_norm;
    ctx->phase = kNormed;
    return TL_OK;
}

int tl_clip_adamw_step(tl_ctx* ctx, const tl_adamw_hp* hp, tl_stream stream) {
    if (ctx == nullptr || hp == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (ctx->phase != kNormed) return fail(ctx, TL_ESTATE, "tl_clip_adamw_step must follow tl_grad_norm");
    if (!(hp->lr >= 0.0f) || !std::isfinite(hp->lr) || !(hp->beta1 >= 0.5f && hp->beta1 < 1.0f) ||
        !(hp->beta2 >= 0.5f && hp->beta2 < 1.0f) || !(hp->eps > 0.0f) || !std::isfinite(hp->eps) ||
        !(hp->weight_decay >= 0.0f) || !std::isfinite(hp->weight_decay))
        return fail(ctx, TL_EINVAL, "AdamW hyper-parameters out of range");
    int rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    AdamHP h{hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, ctx->max_norm, ctx->lr_sched, ctx->lr_len};
    const int pdt = ctx->cfg.param_dtype;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scaler state machine runs in the last CTA of the update's last AdamW launch
    auto scaler = [&](bool last) {
        return ScalerParams{ctx->cfg.scaler_enabled, ctx->cfg.growth, ctx->cfg.backoff, ctx->cfg.interval,
                            ctx->cfg.min_scale, ctx->cfg.max_scale, last ? 1 : 0};
    };
    cudaError_t e = cudaSuccess;
    if (ctx->nchunks == 0) {
        // no elements: still one launch, whose CTA computes the beta powers and runs
        // the scaler
        e = gate(ctx);
        if (e == cudaSuccess) e = launch_adamw(pdt, false, 1, ctx->d_chunks, 0, 0, ctx->d_state, h, scaler(true), 1, s);
        if (e == cudaSuccess) ctx->launches += 1;
    } else if (ctx->remat) {
        // u recomputed from the lists the update was checked on (the same device
        // tables: nothing else has used the cache since)
        static thread_local GradTableMany inl;
        bool by_value = true;
        std::vector<const void* const*> tabs;
        std::vector<GradSlot*> slots;
        const int k = ctx->remat_k;
        if ((rc = resolve_lists(ctx, k, ctx->remat_grads.data(), s, &by_value, tabs, slots)) != TL_OK) return rc;
        ManyArgs a;
        fill_many_args(ctx, ctx->remat_grads.data(), ctx->remat_n, ctx->N_update, 0, k, by_value, tabs, a, inl);
        const int gdt = ctx->cfg.grad_dtype;
        e = over_parts(ctx, [&](bool small, int64_t c0, int64_t c1, bool lastl) {
            return launch_adamw_remat(pdt, gdt, small, ctx->run[small ? 1 : 0], ctx->d_chunks, c0, c1, ctx->d_state, h,
                                      scaler(lastl), inl, a,
                                      ctx->grid_remat[pdt][gdt][k <= kFewLists ? 1 : 0][small ? 1 : 0], s);
        });
        if (e == cudaSuccess)
            for (int i = 0; i < k; ++i) mark_used(slots[size_t(i)], s);
    } else {
        e = over_parts(ctx, [&](bool small, int64_t c0, int64_t c1, bool lastl) {
            return launch_adamw(pdt, small, ctx->run[small ? 1 : 0], ctx->d_chunks, c0, c1, ctx->d_state, h,
                                scaler(lastl),
                                ctx->grid_adam[pdt][small ? 1 : 0], s);
        });
    }
    if (e != cudaSuccess) return launch_fail(ctx, e, "adamw launch");
    ctx->phase = kStepped;
    return TL_OK;
}

int tl_scaler_update(tl_ctx* ctx, tl_stream stream) {
    (void)stream;  // the state machine ran in the last CTA of the AdamW launch
    if (ctx == nullptr) return TL_EINVAL;
    if (int rc0 = refuse_if_interrupted(ctx)) return rc0;
    if (ctx->phase != kStepped) return fail(ctx, TL_ESTATE, "tl_scaler_update must follow tl_clip_adamw_step");
    ctx->phase = kIdle;
    ctx->n_sum = 0;
    ctx->N_update = 0;
    ctx->accumulated = false;
    ctx->remat = false;
    ctx->remat_k = 0;
    ctx->remat_grads.clear();
    return TL_OK;
}

static int read_dev_state(tl_ctx* ctx, DevState* ds, cudaStream_t s) {
    int rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    cudaError_t e = cudaMemcpyAsync(ds, ctx->d_state, sizeof(DevState), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "reading the device scalars");
    return TL_OK;
}

int tl_read_status(tl_ctx* ctx, tl_status* out, tl_stream stream) {
    if (ctx == nullptr || out == nullptr) return TL_EINVAL;
    DevState ds;
    if (ctx->phase == kNormed) {
        // the AdamW launch computes the clip coefficient of the update in flight;
        // a read before it gets the coefficient computed now from the same norm
        int rc0 = check_device(ctx);
        if (rc0 != TL_OK) return rc0;
        cudaError_t e = launch_coef(ctx->d_state, ctx->max_norm, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(ctx, e, "coefficient launch");
    }
    int rc = read_dev_state(ctx, &ds, static_cast<cudaStream_t>(stream));
    if (rc != TL_OK) return rc;
    out->S = ds.S;
    out->count = ds.count;
    out->t = ds.t;
    out->skipped = ds.skipped;
    out->found_inf = ds.found_inf;
    out->norm = ds.norm;
    out->coef = ds.coef;
    out->sumsq = ds.sumsq;
    out->b1p = ds.b1p;
    out->b2p = ds.b2p;
    return TL_OK;
}

int tl_get_state(tl_ctx* ctx, tl_state* out, tl_stream stream) {
    if (ctx == nullptr || out == nullptr) return TL_EINVAL;
    DevState ds;
    int rc = read_dev_state(ctx, &ds, static_cast<cudaStream_t>(stream));
    if (rc != TL_OK) return rc;
    out->S = ds.S;
    out->count = ds.count;
    out->t = ds.t;
    out->b1p = ds.b1p;
    out->b2p = ds.b2p;
    return TL_OK;
}

int tl_set_state(tl_ctx* ctx, const tl_state* in, tl_stream stream) {
    if (ctx == nullptr || in == nullptr) return TL_EINVAL;
    if (ctx->phase != kIdle) return fail(ctx, TL_ESTATE, "tl_set_state is allowed only between updates");
    const tl_config& c = ctx->cfg;
    if (c.scaler_enabled) {
        if (!is_pow2(in->S) || in->S < c.min_scale || in->S > c.max_scale)
            return fail(ctx, TL_EINVAL, "S must be a power of two in [min_scale, max_scale]");
        if (in->count < 0 || in->count >= c.interval) return fail(ctx, TL_EINVAL, "count must be in [0, interval)");
    } else {
        if (in->S != 1.0f || in->count != 0) return fail(ctx, TL_EINVAL, "with the scaler disabled S must be 1 and count 0");
    }
    if (in->t < 0) return fail(ctx, TL_EINVAL, "t must be >= 0");
    if (!(in->b1p > 0.0 && in->b1p <= 1.0) || !(in->b2p > 0.0 && in->b2p <= 1.0))
        return fail(ctx, TL_EINVAL, "beta powers must lie in (0, 1]");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DevState ds;
    int rc = read_dev_state(ctx, &ds, s);
    if (rc != TL_OK) return rc;
    ds.S = in->S;
    ds.count = in->count;
    ds.t = in->t;
    ds.b1p = in->b1p;
    ds.b2p = in->b2p;
    ds.found_inf = 0;
    cudaError_t e = cudaMemcpyAsync(ctx->d_state, &ds, sizeof(DevState), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "writing the device scalars");
    ctx->interrupted = false;
    ctx->remat = false;
    ctx->n_sum = 0;
    ctx->N_update = 0;
    ctx->accumulated = false;
    return TL_OK;
}

int tl_loss_seed(tl_ctx* ctx, int64_t n_i, int64_t N, float* out, tl_stream stream) {
    if (ctx == nullptr) return TL_EINVAL;
    if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 3u) != 0) return fail(ctx, TL_EINVAL, "out must be a 4-byte aligned device address");
    int rc;
    if ((rc = check_counts(ctx, n_i, N)) != TL_OK) return rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    const float w = static_cast<float>(static_cast<double>(n_i) / static_cast<double>(N));
    cudaError_t e = launch_seed(ctx->d_state, w, out, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(ctx, e, "seed launch");
    ctx->launches += 1;
    return TL_OK;
}

int tl_set_lr_schedule(tl_ctx* ctx, const float* lr_table, int64_t len) {
    if (ctx == nullptr) return TL_EINVAL;
    if (len < 0) return fail(ctx, TL_EINVAL, "schedule length must be >= 0");
    if (len == 0) {
        ctx->lr_sched = nullptr;
        ctx->lr_len = 0;
        return TL_OK;
    }
    if (lr_table == nullptr || (reinterpret_cast<uintptr_t>(lr_table) & 3u) != 0)
        return fail(ctx, TL_EINVAL, "schedule must be a 4-byte aligned address");
    int rc;
    if ((rc = check_device(ctx)) != TL_OK) return rc;
    // the kernels read the table: it must be memory the device can address
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, lr_table);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "schedule address");
    bool readable = at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged ||
                    (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr);
    if (at.type == cudaMemoryTypeDevice && at.device != ctx->device) readable = false;
    if (!readable) {
        int pageable = 0;
        if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, ctx->device) !=
            cudaSuccess)
            pageable = 0;
        if (!pageable) return fail(ctx, TL_EINVAL, "schedule must be in memory the device can read");
    }
    ctx->lr_sched = lr_table;
    ctx->lr_len = len;
    return TL_OK;
}

int tl_plan(int64_t ntensors, const int64_t* numel, int32_t sm_count, tl_plan_info* out) {
    if (out == nullptr || ntensors < 0 || ntensors > (int64_t(1) << 31) - 1 || sm_count < 1) return TL_EINVAL;
    if (ntensors > 0 && numel == nullptr) return TL_EINVAL;
    int64_t P = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        if (numel[i] < 0 || numel[i] > (int64_t(1) << 62) / 4 - P) return TL_EINVAL;
        P += numel[i];
    }
    const Plan pl = make_plan(ntensors, numel, sm_count);
    tl_plan_info r{};
    r.nchunks = int64_t(pl.chunks.size());
    r.nbig = pl.nbig;
    r.ngroups = r.nchunks - r.nbig;
    r.seg = pl.seg;
    for (size_t b = size_t(pl.nbig); b < pl.chunks.size(); ++b) r.nsmall += int64_t(pl.chunks[b].segs.size());
    r.run_big = pl.run[0];
    r.run_small = pl.run[1];
    r.split_forms = pl.run[0] > 1 ? 1 : 0;   // the rule of the default build (TL_PAIR_SEGS on)
    r.fused_norm = pl.fuse_norm ? 1 : 0;
    *out = r;
    return TL_OK;
}

int tl_partition(int64_t ntensors, const int64_t* numel, int32_t nranks, int32_t rank, int64_t align,
                 int64_t* tensor, int64_t* start, int64_t* len, int64_t cap, int64_t* count) {
    if (count == nullptr || ntensors < 0 || (ntensors > 0 && numel == nullptr)) return TL_EINVAL;
    *count = 0;
    if (nranks < 1 || rank < 0 || rank >= nranks || align < 1 || cap < 0) return TL_EINVAL;
    int64_t P = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        if (numel[i] < 0 || numel[i] > (int64_t(1) << 62) - P) return TL_EINVAL;
        P += numel[i];
    }
    // boundary b_j: the largest multiple of align not above floor(j * P / nranks),
    // computed without overflow as j * (P / n) + floor(j * (P mod n) / n)
    auto bound = [&](int64_t j) -> int64_t {
        if (j >= nranks) return P;
        const int64_t n = nranks;
        const int64_t f = j * (P / n) + (j * (P % n)) / n;
        return f / align * align;
    };
    const int64_t lo = bound(rank), hi = bound(int64_t(rank) + 1);
    // the tensors that intersect [lo, hi), in tensor order
    int64_t pieces = 0, pos = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        const int64_t a = std::max(lo, pos), b = std::min(hi, pos + numel[i]);
        if (a < b) ++pieces;
        pos += numel[i];
    }
    *count = pieces;
    if (pieces > cap) return TL_EINVAL;
    if (pieces > 0 && (tensor == nullptr || start == nullptr || len == nullptr)) return TL_EINVAL;
    int64_t k = 0;
    pos = 0;
    for (int64_t i = 0; i < ntensors; ++i) {
        const int64_t a = std::max(lo, pos), b = std::min(hi, pos + numel[i]);
        if (a < b) {
            tensor[k] = i;
            start[k] = a - pos;
            len[k] = b - a;
            ++k;
        }
        pos += numel[i];
    }
    return TL_OK;
}

const float* tl_scale_ptr(const tl_ctx* ctx) {
    return ctx == nullptr ? nullptr : &ctx->d_state->S;
}

int64_t tl_num_params(const tl_ctx* ctx) { return ctx == nullptr ? 0 : ctx->P; }
int64_t tl_num_chunks(const tl_ctx* ctx) { return ctx == nullptr ? 0 : ctx->nchunks; }
int64_t tl_launch_count(const tl_ctx* ctx) { return ctx == nullptr ? 0 : ctx->launches; }

}  // extern "C"
