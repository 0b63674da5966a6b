/*
 * tlo.c - the ORACLE for the loss-scaled AdamW optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded CPU
 * statement of what the mixed-precision optimizer step computes.  It exists so
 * that the GPU library can be checked against something written independently
 * of it.  Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load it; the product path never does.  It shares no code,
 * header, table or constant with the CUDA library: every format conversion
 * below is written from the bit layout, and every floating-point operation is
 * an explicit IEEE-754 binary32 (or binary64 where stated) operation.  It must
 * be compiled with -ffp-contract=off and without -ffast-math, so that each
 * '+', '-', '*', '/' and sqrtf() is one correctly rounded operation and the
 * only fused multiply-add is the one written as fmaf().
 *
 * Sources (web pages; cited by title and section):
 *   [MP]   "Mixed precision, loss scaling, gradient accumulation, and activation
 *          checkpointing" (tinyllm module L11.1): section 2 "Principles",
 *          section 3 "Worked example by hand", section 4 "The interface".
 *   [MEG]  "Megatron Internals III: Mixed Precision, Loss Scaling, and Grad
 *          Clipping": section 4 "Loss scaling in one equation", section 5
 *          "Dynamic loss scaling as feedback control", section 8 "Copying
 *          gradients is not just casting", section 9 "Gradient clipping under
 *          model parallelism".
 *   [ZRO]  "Your weights fit on one device but Adam's moments do not - how do
 *          you shard the optimizer state?": sections "Why the optimizer state is
 *          the thing that overflows", "The scheme", "Operational sharp edges"
 *          ("Gradient clipping", "Partition granularity").
 *   [MEG]  also section 6 "Overflow must be global" (the sharded step).
 *   [RST]  "Practical LLM in Rust", chapter 13 "Accumulate gradients and
 *          recompute activations": "Weight each mean by the targets it
 *          represents" (equation block), "Discard a failed partial logical
 *          update".
 *   [T41]  "Training at Scale", chapter 41, section 41.1, equation (41.1).
 *
 * Readings where the pages leave a step open (each one is applied in exactly
 * one place below and marked READING):
 *   R1  backoff multiplies S by 1/2 ([MP] "Dynamic scaling"; [MEG] section 5
 *       prints a division by the backoff factor, read as the same halving);
 *   R2  min_scale floors S after backoff, max_scale caps it after growth;
 *   R3  clip coefficient = max_norm / (norm + 1e-6), applied only when < 1;
 *   R4  the squared norm sums the fp32 squares fl32(u*u) in fp64, tensor order
 *       then element order; a non-finite sum is treated as an overflow;
 *   R5  a skipped step advances neither t nor the good-step count;
 *   R6  AdamW: eps outside the square root, decoupled decay lr*wd applied to
 *       the pre-update master, bias corrections from fp64 beta powers;
 *   R7  with the scaler disabled (bf16), S stays fixed, count stays 0, and the
 *       finite check still gates the step;
 *   R17 8-bit gradients: [T41] section 41.5 names E4M3 but does not print its
 *       emulator; the OCP E4M3 layout is taken (bias 7, 3 mantissa bits,
 *       subnormals, no infinity, S.1111.111 is NaN, largest finite 448);
 *   R18 block scales run over each tensor's flattened elements in blocks of 16
 *       (the section's block_size), and a tensor's last block may hold fewer
 *       than 16 elements.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <stdlib.h>

#define TLO_DT_F32 0
#define TLO_DT_BF16 1
#define TLO_DT_F16 2
#define TLO_DT_E4M3B16 3

/* ------------------------------------------------------------------------ */
/* 16-bit formats.  [MP] section 2 "Two 16-bit formats": bf16 keeps fp32's   */
/* 8 exponent bits and 7 mantissa bits; fp16 has 5 exponent bits and 10      */
/* mantissa bits, largest finite 65504, smallest normal 2^-14, smallest      */
/* subnormal 2^-24.  rd16 rounds to nearest, ties to even.                   */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }
static float bits_f32(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }

float tlo_bf16_to_f32(uint16_t h) {
    /* bf16 is the upper half of an fp32 word. */
    return bits_f32((uint32_t)h << 16);
}

float tlo_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    float mag;
    if (exp == 0) {
        mag = ldexpf((float)man, -24);                 /* zero or subnormal: man * 2^-24 */
    } else if (exp == 31) {
        mag = man ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(1024 + man), exp - 25);   /* (1.man) * 2^(exp-15) */
    }
    return sign ? -mag : mag;
}

/* Round the non-negative integer sig / 2^shift to the nearest integer, ties
 * to even.  shift >= 1. */
static uint32_t rne_shift(uint32_t sig, int shift) {
    if (shift > 31) return 0;                           /* sig < 2^24 < half */
    uint32_t kept = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u))) kept += 1u;
    return kept;
}

uint16_t tlo_f32_to_bf16(float f) {
    uint32_t b = f32_bits(f);
    uint32_t a = b & 0x7fffffffu;
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7fc0u);   /* NaN stays NaN */
    /* Keep the top 16 bits, rounding the dropped 16 bits to nearest even.  A
     * carry out of the mantissa increments the exponent, which is the correct
     * next bf16 value (up to infinity). */
    uint32_t kept = a >> 16;
    uint32_t rem = a & 0xffffu;
    if (rem > 0x8000u || (rem == 0x8000u && (kept & 1u))) kept += 1u;
    return (uint16_t)(sign | kept);
}

uint16_t tlo_f32_to_f16(float f) {
    uint32_t b = f32_bits(f);
    uint32_t a = b & 0x7fffffffu;
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);   /* NaN */
    if (a == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);  /* inf */
    if (a == 0) return sign;
    /* |f| = sig * 2^(e - 23) with a 24-bit significand sig. */
    int e;
    uint32_t sig;
    if (a >= 0x00800000u) { e = (int)(a >> 23) - 127; sig = (a & 0x7fffffu) | 0x800000u; }
    else                  { e = -126;                 sig = a; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);            /* >= 2^16: overflows */
    if (e >= -14) {
        /* Normal fp16 range: keep 11 significant bits (drop 13). */
        uint32_t kept = rne_shift(sig, 13);                    /* in [1024, 2048] */
        int ee = e;
        if (kept == 2048u) { kept = 1024u; ee += 1; }
        if (ee > 15) return (uint16_t)(sign | 0x7c00u);        /* rounded past 65504 */
        return (uint16_t)(sign | (uint16_t)((ee + 15) << 10) | (uint16_t)(kept - 1024u));
    }
    /* Subnormal fp16: the value in units of 2^-24, rounded to nearest even.
     * sig * 2^(e-23) / 2^-24 = sig / 2^(-1 - e).  A result of 1024 is the
     * smallest normal 2^-14, whose encoding is exactly 0x0400. */
    uint32_t units = rne_shift(sig, -1 - e);
    return (uint16_t)(sign | units);
}

/* Array forms of the conversions above. */
void tlo_decode16(const uint16_t* h, float* out, int64_t n, int dtype) {
    for (int64_t j = 0; j < n; ++j)
        out[j] = (dtype == TLO_DT_F16) ? tlo_f16_to_f32(h[j]) : tlo_bf16_to_f32(h[j]);
}

void tlo_recast(const float* x, uint16_t* out, int64_t n, int dtype) {
    for (int64_t j = 0; j < n; ++j)
        out[j] = (dtype == TLO_DT_F16) ? tlo_f32_to_f16(x[j]) : tlo_f32_to_bf16(x[j]);
}

/* ------------------------------------------------------------------------ */
/* 8-bit gradients with fine-grained scaling.  [T41] section 41.5 "FP8       */
/* training with fine-grained scaling": one scale per block of values, the   */
/* values stored in E4M3 relative to that scale and dequantized (code value  */
/* times block scale) before accumulation.  READING R17 fixes the format.    */
/* ------------------------------------------------------------------------ */
float tlo_e4m3_to_f32(uint8_t c) {
    const uint32_t sign = (uint32_t)(c >> 7) << 31;
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 15u && m == 7u) return bits_f32(sign | 0x7FC00000u);    /* NaN */
    if (e == 0u) {
        /* subnormal: m * 2^-9, an exact product of a small integer and a power of two */
        const float mag = (float)m * (1.0f / 512.0f);
        return bits_f32(sign | f32_bits(mag));
    }
    /* normal: (1 + m/8) * 2^(e-7); binary32 exponent field e - 7 + 127, mantissa m in its top 3 bits */
    return bits_f32(sign | ((e + 120u) << 23) | (m << 20));
}

/* The gradients of one micro-batch as E4M3 codes plus fp32 block scales: the
 * codes of every tensor back to back (tensor order), and each tensor's
 * ceil(numel/16) scales back to back (READING R18). */
typedef struct {
    const uint8_t* codes;
    const float* scales;
    const int64_t* numel;
    int64_t ntensors;
} tlo_e4m3_list;

/* g[j] = fl32(e4m3(code[j]) * scale of j's block) over the whole list. */
void tlo_dequant_e4m3b16(const tlo_e4m3_list* g, float* out) {
    int64_t j = 0, b = 0;
    for (int64_t t = 0; t < g->ntensors; ++t) {
        for (int64_t e = 0; e < g->numel[t]; ++e, ++j)
            out[j] = tlo_e4m3_to_f32(g->codes[j]) * g->scales[b + e / 16];
        b += (g->numel[t] + 15) / 16;
    }
}

static float load_grad(const void* g, int dtype, int64_t j) {
    if (dtype == TLO_DT_BF16) return tlo_bf16_to_f32(((const uint16_t*)g)[j]);
    if (dtype == TLO_DT_F16) return tlo_f16_to_f32(((const uint16_t*)g)[j]);
    return ((const float*)g)[j];
}

/* ------------------------------------------------------------------------ */
/* Token weighting.  [RST] "Weight each mean by the targets it represents":  */
/* N = sum n_i, L = sum (n_i/N) L_i, so micro-batch i's gradient is weighted */
/* by n_i/N; [MP] section 2 "Gradient accumulation" gives the same identity. */
/* The integers convert exactly to fp64 (N <= 2^53); the quotient is rounded */
/* once to fp32.                                                              */
/* ------------------------------------------------------------------------ */
float tlo_microbatch_weight(int64_t n_i, int64_t N) {
    return (float)((double)n_i / (double)N);
}

/* Accumulate micro-batch gradient g (P elements) into the fp32 buffer acc:
 * acc = w*g for the first micro-batch, acc = fma(w, g, acc) afterwards.  No
 * zeroing in between ([MP] section 2 "Gradient accumulation"); the fp32
 * buffer is the master-gradient buffer of [MEG] section 8. */
void tlo_accumulate(float* acc, const void* g, int gdtype, int64_t P, float w, int first) {
    for (int64_t j = 0; j < P; ++j) {
        float gj = load_grad(g, gdtype, j);
        if (first) acc[j] = w * gj;
        else acc[j] = fmaf(w, gj, acc[j]);
    }
}

/* Unscale by 1/S and check.  [MEG] section 4: grad = scaled_grad / S; [MP]
 * section 2 "Loss scaling": with S a power of two the division only changes
 * the exponent.  [MEG] section 6 / [MP] "Dynamic scaling": any non-finite
 * gradient flags the whole step.  u overwrites acc.  Returns found_inf. */
int tlo_unscale_check(float* acc, int64_t P, float S) {
    float inv_s = 1.0f / S;
    int found_inf = 0;
    for (int64_t j = 0; j < P; ++j) {
        float u = acc[j] * inv_s;
        acc[j] = u;
        if (!isfinite(u)) found_inf = 1;
    }
    return found_inf;
}

/* Global squared L2 norm.  [MEG] section 9: global_norm = sqrt(sum_i
 * ||grad_i||^2).  READING R4: each square is the fp32 product u*u, summed in
 * fp64 in element order of the flattened list (tensor order, then element
 * order). */
double tlo_sumsq(const float* u, int64_t P) {
    double s = 0.0;
    for (int64_t j = 0; j < P; ++j) {
        float sq = u[j] * u[j];
        s += (double)sq;
    }
    return s;
}

float tlo_norm_from_sumsq(double sumsq) {
    return (float)sqrt(sumsq);
}

/* [MEG] section 9: clip_coef = max_norm / (global_norm + eps).  READING R3:
 * eps = 1e-6 and the gradient is scaled only when the coefficient is below 1;
 * max_norm <= 0 disables clipping.  [MP] "Dynamic scaling": clipping happens
 * after unscaling, so norm is in true gradient units. */
float tlo_clip_coef(float norm, float max_norm) {
    if (!(max_norm > 0.0f)) return 1.0f;
    float c = max_norm / (norm + 1e-6f);
    return c < 1.0f ? c : 1.0f;
}

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} tlo_adamw_hp;

/* The learning rate a schedule gives the update that would commit optimizer
 * step t+1, where t counts the committed steps only: [RST] "Discard a failed
 * partial logical update" (a skipped attempt leaves the optimizer step where it
 * was and the next scheduled step still available) and "Carry one logical update
 * into schedule reasoning" (warm-up and decay are stated per logical update).
 * table[i] is the rate of optimizer step i+1; past the end of the table the last
 * entry holds. */
float tlo_scheduled_lr(const float* table, int64_t len, int64_t t) {
    return table[t < len ? t : len - 1];
}

/* The per-step scalars of AdamW for the step about to be committed (t+1),
 * computed in fp64 from the beta powers kept as state ([RST] "Discard a
 * failed partial logical update": the optimizer state includes the beta
 * powers) and rounded once to fp32. */
typedef struct {
    float step_size;   /* lr / (1 - beta1^(t+1)) */
    float bc2_sqrt;    /* sqrt(1 - beta2^(t+1)) */
    float lr_wd;       /* lr * weight_decay */
    float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
} tlo_adamw_scalars;

tlo_adamw_scalars tlo_adamw_prepare(const tlo_adamw_hp* hp, double b1p_next, double b2p_next) {
    tlo_adamw_scalars s;
    s.step_size = (float)((double)hp->lr / (1.0 - b1p_next));
    s.bc2_sqrt = (float)sqrt(1.0 - b2p_next);
    s.lr_wd = (float)((double)hp->lr * (double)hp->weight_decay);
    s.beta1 = hp->beta1;
    s.one_minus_beta1 = 1.0f - hp->beta1;
    s.beta2 = hp->beta2;
    s.one_minus_beta2 = 1.0f - hp->beta2;
    s.eps = hp->eps;
    return s;
}

/* Clip + AdamW on the fp32 masters + recast ([MEG] sections 7 and 9: clip
 * local gradients with the global coefficient, step fp32 master parameters,
 * copy master parameters back to model precision; [ZRO] "Why the optimizer
 * state...": the update divides the bias-corrected first moment by the
 * square root of the bias-corrected second moment plus a small constant;
 * [RST] "Weight each mean...": decoupled weight decay; READING R6 fixes the
 * form).  pdtype selects bf16 or fp16 for the model copy p. */
void tlo_adamw_recast(float* w, float* m, float* v, uint16_t* p, int pdtype,
                      const float* u, int64_t P, float coef, const tlo_adamw_scalars* s) {
    for (int64_t j = 0; j < P; ++j) {
        float g = u[j] * coef;
        float mj = s->beta1 * m[j] + s->one_minus_beta1 * g;
        float vj = s->beta2 * v[j] + s->one_minus_beta2 * (g * g);
        float wj = w[j];
        wj = wj - s->lr_wd * wj;
        float denom = sqrtf(vj) / s->bc2_sqrt + s->eps;
        wj = wj - s->step_size * (mj / denom);
        m[j] = mj;
        v[j] = vj;
        w[j] = wj;
        /* [MP] section 2 "Why the weights stay float32": only the model copy
         * is rounded; the master keeps the update. */
        p[j] = (pdtype == TLO_DT_F16) ? tlo_f32_to_f16(wj) : tlo_f32_to_bf16(wj);
    }
}

/* ------------------------------------------------------------------------ */
/* The dynamic loss scaler.  [MEG] section 5 controller; [MP] "Dynamic        */
/* scaling" and section 3's five-step trace; [RST] "Discard a failed partial */
/* logical update": a skipped attempt leaves weights, moments, beta powers   */
/* and the optimizer step unchanged.                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    int enabled;       /* 0: bf16 mode, READING R7 */
    float growth;      /* 2 */
    float backoff;     /* 1/2, READING R1 */
    int32_t interval;  /* good steps between growths */
    float min_scale;   /* READING R2 */
    float max_scale;
} tlo_scaler_cfg;

typedef struct {
    float S;           /* loss scale */
    int32_t count;     /* good steps since the last overflow or growth */
    int64_t t;         /* committed optimizer steps */
    double b1p, b2p;   /* beta1^t, beta2^t */
} tlo_state;

void tlo_scaler_update(tlo_state* st, const tlo_scaler_cfg* cfg, int found_inf,
                       double b1p_next, double b2p_next) {
    if (found_inf) {
        if (cfg->enabled) {
            float s = st->S * cfg->backoff;
            st->S = s > cfg->min_scale ? s : cfg->min_scale;
        }
        st->count = 0;
        return;                                   /* READING R5 */
    }
    st->t += 1;
    st->b1p = b1p_next;
    st->b2p = b2p_next;
    if (cfg->enabled) {
        st->count += 1;
        if (st->count == cfg->interval) {
            float s = st->S * cfg->growth;
            st->S = s < cfg->max_scale ? s : cfg->max_scale;
            st->count = 0;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* One attempted logical update, in the order of [MEG] section 9 ("The order */
/* matters"): accumulate the k micro-batches, unscale, detect overflow, take */
/* the global norm, clip, step fp32 masters, copy back, update the scaler.   */
/* grads[i] points at micro-batch i's P gradient values of type gdtype.      */
/* acc is caller-provided scratch of P floats.                                */
/* ------------------------------------------------------------------------ */
typedef struct {
    int skipped;
    int found_inf;
    float norm;
    float coef;
    double sumsq;
} tlo_result;

int tlo_step(float* w, float* m, float* v, uint16_t* p, int pdtype, float* acc, int64_t P,
             const void* const* grads, int gdtype, const int64_t* counts, int k,
             float max_norm, const tlo_adamw_hp* hp, const tlo_scaler_cfg* cfg,
             tlo_state* st, tlo_result* res) {
    if (k < 1) return -1;
    int64_t N = 0;
    for (int i = 0; i < k; ++i) {
        if (counts[i] <= 0) return -1;
        N += counts[i];
    }
    if (N > ((int64_t)1 << 53)) return -1;
    float* deq = NULL;
    if (gdtype == TLO_DT_E4M3B16) {
        deq = (float*)malloc(sizeof(float) * (size_t)(P > 0 ? P : 1));
        if (deq == NULL) return -1;
    }
    for (int i = 0; i < k; ++i) {
        const void* gi = grads[i];
        int gdt = gdtype;
        if (deq != NULL) {  /* 8-bit gradients: dequantize, then accumulate the fp32 values */
            tlo_dequant_e4m3b16((const tlo_e4m3_list*)grads[i], deq);
            gi = deq;
            gdt = TLO_DT_F32;
        }
        tlo_accumulate(acc, gi, gdt, P, tlo_microbatch_weight(counts[i], N), i == 0);
    }
    free(deq);
    int found_inf = tlo_unscale_check(acc, P, st->S);
    double sumsq = 0.0;
    float norm = 0.0f, coef = 1.0f;
    if (!found_inf) {
        sumsq = tlo_sumsq(acc, P);
        if (!isfinite(sumsq)) found_inf = 1;       /* READING R4 */
        norm = tlo_norm_from_sumsq(sumsq);
        coef = tlo_clip_coef(norm, max_norm);
    }
    double b1p_next = st->b1p * (double)hp->beta1;
    double b2p_next = st->b2p * (double)hp->beta2;
    if (!found_inf) {
        tlo_adamw_scalars s = tlo_adamw_prepare(hp, b1p_next, b2p_next);
        tlo_adamw_recast(w, m, v, p, pdtype, acc, P, coef, &s);
    }
    tlo_scaler_update(st, cfg, found_inf, b1p_next, b2p_next);
    res->skipped = found_inf;
    res->found_inf = found_inf;
    res->norm = norm;
    res->coef = coef;
    res->sumsq = sumsq;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The sharded step.  [ZRO] "The scheme": the parameter vector is split into  */
/* N disjoint slices and device i keeps the master weights and both moments  */
/* of slice i alone and updates that slice; "Partition granularity": slicing */
/* the flat vector may split a tensor between owners.  [ZRO] "Operational    */
/* sharp edges", "Gradient clipping": each device sums the squares over its  */
/* own slice and those scalars are all-reduced before the root is taken.     */
/* [MEG] section 6 "Overflow must be global": the overflow flag is           */
/* all-reduced with max, so every rank steps or skips together; section 9:   */
/* local squared norms, reduced, then one coefficient for every rank.        */
/* ------------------------------------------------------------------------ */

/* Cut points of nranks slices of a flattened list of P elements (tensor order,
 * then element order): bounds[j] = the largest multiple of align that is not
 * above floor(j * P / nranks), for j < nranks, and bounds[nranks] = P.  Slice r
 * is [bounds[r], bounds[r+1]). */
void tlo_partition_bounds(int64_t P, int nranks, int64_t align, int64_t* bounds) {
    for (int j = 0; j < nranks; ++j) {
        __int128 f = ((__int128)j * (__int128)P) / (__int128)nranks;
        bounds[j] = (int64_t)(f - f % (__int128)align);
    }
    bounds[nranks] = P;
}

static int64_t elem_bytes(int dtype) {
    return dtype == TLO_DT_F32 ? 4 : 2;
}

/* One attempted logical update of a list sharded over nranks owners, every rank
 * simulated in turn: each rank accumulates, unscales and checks its own slice
 * and sums its own squares (rank_flag[r], rank_sumsq[r]); the flags are combined
 * with max and the squared norms summed in rank order (the all-reduces); every
 * rank then clips with the one global coefficient and steps its slice, and the
 * scaler takes the global decision once.  Same arguments as tlo_step plus the
 * slicing (nranks >= 1, align >= 1) and the per-rank outputs. */
int tlo_step_sharded(float* w, float* m, float* v, uint16_t* p, int pdtype, float* acc, int64_t P,
                     const void* const* grads, int gdtype, const int64_t* counts, int k,
                     float max_norm, const tlo_adamw_hp* hp, const tlo_scaler_cfg* cfg,
                     tlo_state* st, tlo_result* res, int nranks, int64_t align,
                     double* rank_sumsq, int* rank_flag) {
    if (k < 1 || nranks < 1 || align < 1) return -1;
    int64_t N = 0;
    for (int i = 0; i < k; ++i) {
        if (counts[i] <= 0) return -1;
        N += counts[i];
    }
    if (N > ((int64_t)1 << 53)) return -1;
    int64_t* b = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nranks + 1));
    if (b == NULL) return -1;
    tlo_partition_bounds(P, nranks, align, b);
    float* deq = NULL;
    if (gdtype == TLO_DT_E4M3B16) {
        deq = (float*)malloc(sizeof(float) * (size_t)(P > 0 ? P : 1));
        if (deq == NULL) { free(b); return -1; }
    }
    /* every rank accumulates its slice of every micro-batch */
    for (int i = 0; i < k; ++i) {
        const char* gi = (const char*)grads[i];
        int gdt = gdtype;
        if (deq != NULL) {
            tlo_dequant_e4m3b16((const tlo_e4m3_list*)grads[i], deq);
            gi = (const char*)deq;
            gdt = TLO_DT_F32;
        }
        float wi = tlo_microbatch_weight(counts[i], N);
        for (int r = 0; r < nranks; ++r)
            tlo_accumulate(acc + b[r], gi + b[r] * elem_bytes(gdt), gdt, b[r + 1] - b[r], wi, i == 0);
    }
    free(deq);
    /* local unscale, check and squared norm of each slice */
    for (int r = 0; r < nranks; ++r) {
        rank_flag[r] = tlo_unscale_check(acc + b[r], b[r + 1] - b[r], st->S);
        rank_sumsq[r] = tlo_sumsq(acc + b[r], b[r + 1] - b[r]);
    }
    /* the all-reduces: max of the flags, sum of the squared norms in rank order */
    int found_inf = 0;
    double sumsq = 0.0;
    for (int r = 0; r < nranks; ++r) {
        if (rank_flag[r]) found_inf = 1;
        sumsq += rank_sumsq[r];
    }
    float norm = 0.0f, coef = 1.0f;
    if (!found_inf) {
        found_inf = isfinite(sumsq) ? 0 : 1;        /* READING R4 */
        norm = tlo_norm_from_sumsq(sumsq);
        coef = tlo_clip_coef(norm, max_norm);
    } else {
        sumsq = 0.0;
    }
    const double b1n = (double)hp->beta1 * st->b1p;   /* beta powers of step t+1 */
    const double b2n = (double)hp->beta2 * st->b2p;
    if (found_inf == 0) {   /* every rank steps its own slice with the one coefficient */
        const tlo_adamw_scalars s = tlo_adamw_prepare(hp, b1n, b2n);
        for (int r = 0; r < nranks; ++r)
            tlo_adamw_recast(w + b[r], m + b[r], v + b[r], p + b[r], pdtype, acc + b[r], b[r + 1] - b[r], coef, &s);
    }
    tlo_scaler_update(st, cfg, found_inf, b1n, b2n);
    free(b);
    res->skipped = found_inf;
    res->found_inf = found_inf;
    res->norm = norm;
    res->coef = coef;
    res->sumsq = sumsq;
    return 0;
}
