"""Mutation check of the oracle's pins: each planted mistake below (a dropped
term, a wrong sign, a swapped operand, an off-by-one, and the pitfalls the
mixed-precision page lists as s07-s15) is compiled into a copy of the oracle on
the CPU, and at least one pin must fail against it.  The real oracle is never
modified."""
import os
import shutil
import tempfile

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "tlo.c")

# (name, original text, mutated text): each original must occur exactly once.
MUTANTS = [
    # [MP] pitfalls 7-9: 1/k weighting, summing, zeroing between micro-batches
    ("s07_one_over_k", "tlo_microbatch_weight(counts[i], N), i == 0)", "1.0f / (float)k, i == 0)"),
    ("s08_sum_losses", "tlo_microbatch_weight(counts[i], N), i == 0)", "1.0f, i == 0)"),
    ("s09_zero_between", "tlo_microbatch_weight(counts[i], N), i == 0)", "tlo_microbatch_weight(counts[i], N), 1)"),
    ("weight_swapped", "return (float)((double)n_i / (double)N);", "return (float)((double)N / (double)n_i);"),
    ("acc_no_fma_weight", "else acc[j] = fmaf(w, gj, acc[j]);", "else acc[j] = gj + acc[j];"),
    # [MP] pitfall 11: never unscaling; pitfall 12: stepping on non-finite
    ("s11_no_unscale", "float u = acc[j] * inv_s;", "float u = acc[j];"),
    ("unscale_multiplies", "float inv_s = 1.0f / S;", "float inv_s = S;"),
    ("s12_step_on_inf", "        if (!isfinite(u)) found_inf = 1;\n", "\n"),
    # [MP] pitfall 13: keeping the bad gradients after a skip
    ("s13_keep_bad_grads", "tlo_microbatch_weight(counts[i], N), i == 0)", "tlo_microbatch_weight(counts[i], N), 0)"),
    # [MP] pitfall 14: not restarting the count after an overflow
    ("s14_count_not_reset", "        st->count = 0;\n        return;", "        return;"),
    # [MP] pitfall 15: clipping before unscaling
    ("s15_clip_before_unscale", "int found_inf = tlo_unscale_check(acc, P, st->S);",
     "double pre = tlo_sumsq(acc, P); int found_inf = tlo_unscale_check(acc, P, st->S); (void)pre;"
     " if (!found_inf) { float sc = st->S; for (int64_t j = 0; j < P; ++j) acc[j] *= sc; }"),
    # scaler slips
    ("no_backoff", "float s = st->S * cfg->backoff;", "float s = st->S;"),
    ("growth_off_by_one", "if (st->count == cfg->interval) {", "if (st->count + 1 == cfg->interval) {"),
    ("t_advances_on_skip", "        st->count = 0;\n        return;",
     "        st->count = 0;\n        st->t += 1; st->b1p = b1p_next; st->b2p = b2p_next;\n        return;"),
    ("min_scale_ignored", "st->S = s > cfg->min_scale ? s : cfg->min_scale;", "st->S = s;"),
    # norm / clip slips
    ("sumsq_abs", "float sq = u[j] * u[j];", "float sq = fabsf(u[j]);"),
    ("norm_no_sqrt", "return (float)sqrt(sumsq);", "return (float)sumsq;"),
    ("clip_not_clamped", "return c < 1.0f ? c : 1.0f;", "return c;"),
    ("clip_inverted", "float c = max_norm / (norm + 1e-6f);", "float c = (norm + 1e-6f) / max_norm;"),
    ("nonfinite_norm_ignored", "if (!isfinite(sumsq)) found_inf = 1;", ";"),
    # AdamW slips: bias corrections, eps placement, decay, swapped betas, wrong moments
    ("no_bias_correction1", "s.step_size = (float)((double)hp->lr / (1.0 - b1p_next));", "s.step_size = hp->lr;"),
    ("no_bias_correction2", "s.bc2_sqrt = (float)sqrt(1.0 - b2p_next);", "s.bc2_sqrt = 1.0f;"),
    ("bias_correction_old_t", "double b1p_next = st->b1p * (double)hp->beta1;", "double b1p_next = st->b1p == 1.0 ? 0.5 : st->b1p;"),
    ("eps_inside_sqrt", "float denom = sqrtf(vj) / s->bc2_sqrt + s->eps;", "float denom = sqrtf(vj / (s->bc2_sqrt * s->bc2_sqrt) + s->eps);"),
    ("decay_sign", "wj = wj - s->lr_wd * wj;", "wj = wj + s->lr_wd * wj;"),
    ("decay_after_update", "        wj = wj - s->lr_wd * wj;\n", "\n"),
    ("decay_not_times_lr", "s.lr_wd = (float)((double)hp->lr * (double)hp->weight_decay);", "s.lr_wd = hp->weight_decay;"),
    ("betas_swapped", "s.beta1 = hp->beta1;", "s.beta1 = hp->beta2;"),
    ("m_uses_g_squared", "float mj = s->beta1 * m[j] + s->one_minus_beta1 * g;", "float mj = s->beta1 * m[j] + s->one_minus_beta1 * (g * g);"),
    ("v_uses_g", "s->one_minus_beta2 * (g * g);", "s->one_minus_beta2 * g;"),
    ("update_sign", "wj = wj - s->step_size * (mj / denom);", "wj = wj + s->step_size * (mj / denom);"),
    # schedule slips: a rate one step ahead, or the first rate for every step
    ("schedule_off_by_one", "return table[t < len ? t : len - 1];", "return table[t + 1 < len ? t + 1 : len - 1];"),
    ("schedule_first_only", "return table[t < len ? t : len - 1];", "return table[0];"),
    ("clip_coef_unused", "float g = u[j] * coef;", "float g = u[j];"),
    # recast / formats
    ("bf16_truncates", "if (rem > 0x8000u || (rem == 0x8000u && (kept & 1u))) kept += 1u;\n    return (uint16_t)(sign | kept);",
     "return (uint16_t)(sign | kept);"),
    ("rne_ties_up", "if (rem > half || (rem == half && (kept & 1u))) kept += 1u;", "if (rem >= half) kept += 1u;"),
    ("f16_bias_off", "mag = ldexpf((float)(1024 + man), exp - 25);", "mag = ldexpf((float)(1024 + man), exp - 24);"),
    ("f16_subnormal_scale", "mag = ldexpf((float)man, -24);", "mag = ldexpf((float)man, -25);"),
    ("param_not_recast", "p[j] = (pdtype == TLO_DT_F16) ? tlo_f32_to_f16(wj) : tlo_f32_to_bf16(wj);", "(void)p;"),
    # [MP] pitfall 16: losing the good-step count; pitfall 17: stepping on a NaN without a scaler
    ("s16_count_lost", "        st->count += 1;\n", "        st->count = 1;\n"),
    ("s17_nan_without_scaler", "    if (!found_inf) {\n        tlo_adamw_scalars s",
     "    if (!found_inf || !cfg->enabled) {\n        tlo_adamw_scalars s"),
    # 8-bit gradients: E4M3 layout and block scales
    ("e4m3_bias_off", "((e + 120u) << 23)", "((e + 121u) << 23)"),
    ("e4m3_mantissa_shift", "| (m << 20));", "| (m << 21));"),
    ("e4m3_subnormal_scale", "(float)m * (1.0f / 512.0f);", "(float)m * (1.0f / 1024.0f);"),
    ("e4m3_no_nan", "if (e == 15u && m == 7u) return bits_f32(sign | 0x7FC00000u);", ";"),
    ("e4m3_sign_dropped", "const uint32_t sign = (uint32_t)(c >> 7) << 31;", "const uint32_t sign = 0u;"),
    ("block_index_over_list", "g->scales[b + e / 16];", "g->scales[j / 16];"),
    ("block_size_8", "g->scales[b + e / 16];", "g->scales[b + e / 8];"),
    ("scale_not_applied", "out[j] = tlo_e4m3_to_f32(g->codes[j]) * g->scales[b + e / 16];",
     "out[j] = tlo_e4m3_to_f32(g->codes[j]);"),
    # the sharded step: a rank's squares left out of the sum, each rank clipping with its
    # own partial norm ([ZRO] "Gradient clipping" warns of exactly this), and cuts off the
    # alignment.  (A flag combined from one rank only is no mistake the pins can see: a
    # non-finite element makes its square, hence the all-reduced sum, non-finite, and the
    # non-finite sum skips the update on every rank anyway.)
    ("shard_sum_drops_rank", "        sumsq += rank_sumsq[r];\n", "        if (r > 0) sumsq += rank_sumsq[r];\n"),
    ("shard_local_clip", "b[r + 1] - b[r], coef, &s);",
     "b[r + 1] - b[r], tlo_clip_coef(tlo_norm_from_sumsq(rank_sumsq[r]), max_norm), &s);"),
    ("shard_cut_unaligned", "bounds[j] = (int64_t)(f - f % (__int128)align);", "bounds[j] = (int64_t)f;"),
]


def _fails(lib):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception:  # any failure or error counts as the mutant being caught
            failed.append(pin.__name__)
    return failed


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="tlo_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} must occur once"
    mpath = os.path.join(workdir, f"{name}.c")
    with open(mpath, "w") as fh:
        fh.write(src.replace(old, new))
    lib = oracle.load(oracle.compile_library(mpath, os.path.join(workdir, f"{name}.so")))
    assert _fails(lib), f"no pin catches mutant {name}"
