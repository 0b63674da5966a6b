"""Pins of the oracle to facts outside itself.

Every function here takes a loaded oracle library (``oracle.load()`` or a
deliberately mutated build of it) and raises AssertionError when the oracle
disagrees with a fact fixed by the pages or by mathematics: a worked example
printed on a page (fixtures under tests/golden/, each carrying its citation), a
closed form, an invariant, a textbook special case, or an independent library
routine (torch.optim.AdamW, torch.nn.utils.clip_grad_norm_, numpy/torch
16-bit conversions).  tests/test_oracle_pins.py runs them against the real
oracle; tests/test_oracle_mutants.py runs them against planted mistakes and
requires each mistake to be caught.

Pages cited (by title):
  [MP]  "Mixed precision, loss scaling, gradient accumulation, and activation
        checkpointing" (tinyllm L11.1)
  [MEG] "Megatron Internals III: Mixed Precision, Loss Scaling, and Grad Clipping"
  [ZRO] "Your weights fit on one device but Adam's moments do not - how do you
        shard the optimizer state?"
  [RST] "Practical LLM in Rust", ch. 13 "Accumulate gradients and recompute activations"
  [T41] "Training at Scale", ch. 41
"""
from __future__ import annotations

import ctypes
import math
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F32_EPS = 2.0 ** -24  # unit roundoff of binary32


def read_golden(name: str):
    """Parse a golden fixture: 'key = value' lines and bare table rows."""
    kv, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
            else:
                rows.append(line.split())
    return kv, rows


def num(s: str) -> float:
    """Parse '7/3', '2^-24', 'inf' or a decimal."""
    s = s.strip()
    if s == "inf":
        return math.inf
    if "^" in s:
        b, e = s.split("^")
        return float(b) ** float(e)
    return float(Fraction(s))


def ulp32(x: float) -> float:
    x = abs(float(np.float32(x)))
    return float(np.spacing(np.float32(x)))


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def make_oracle(lib, master, pdtype="bf16", gdtype="f32", **kw):
    master = np.asarray(master, dtype=np.float32)
    pbits = np.empty(master.size, np.uint16)
    lib.tlo_recast(_p(master), _p(pbits), master.size, oracle.dtype_code(pdtype))
    return oracle.Oracle(master, pbits, param_dtype=pdtype, grad_dtype=gdtype, lib=lib, **kw)


def accumulated_u(lib, grads, counts, S=None):
    """u after one logical update with the optimizer frozen (lr = wd = 0)."""
    P = np.asarray(grads[0]).size
    kw = {} if S is None else {"scaler_enabled": True, "init_scale": S, "interval": 10 ** 6}
    o = make_oracle(lib, np.zeros(P, np.float32), gdtype="f32", **kw)
    res = o.step([np.asarray(g, np.float32) for g in grads], counts, max_norm=0.0, lr=0.0, weight_decay=0.0)
    return o.acc.copy(), res


# --------------------------------------------------------------------------
# Token weighting and accumulation
# --------------------------------------------------------------------------

def pin_weighted_mean_7_3(lib):
    """[RST] ch. 13 constructed example: means 1 and 3 over 2 and 4 targets give 7/3, not 2."""
    kv, _ = read_golden("weighting_examples.txt")
    counts = [int(c) for c in kv["mean_example.counts"].split()]
    means = [num(x) for x in kv["mean_example.means"].split()]
    u, _ = accumulated_u(lib, [[means[0]], [means[1]]], counts)
    want = num(kv["mean_example.weighted"])
    assert abs(u[0] - want) <= ulp32(want), (u[0], want)
    assert abs(u[0] - num(kv["mean_example.equal_weights"])) > 0.3


def pin_hand_example_gradient_minus_15(lib):
    """[MP] section 3 Accumulation table: -2 (1 row) and -58/3 (3 rows) weighted give -15."""
    kv, _ = read_golden("weighting_examples.txt")
    counts = [int(c) for c in kv["grad_example.counts"].split()]
    grads = [np.float32(num(x)) for x in kv["grad_example.grads"].split()]
    u, _ = accumulated_u(lib, [[grads[0]], [grads[1]]], counts)
    want = num(kv["grad_example.weighted"])
    assert abs(u[0] - want) <= 2 * ulp32(want), (u[0], want)
    for wrong in ("grad_example.half_weights", "grad_example.unweighted"):
        assert abs(u[0] - num(kv[wrong])) > 1.0


def pin_backward_seed_shares(lib):
    """[RST] ch. 13: S*6/9 = 85.33333333333333 and S*3/9 = 42.666666666666664 at S = 128.
    The oracle's fp32 weight n_i/N times the power-of-two S is the fp32 rounding of that seed."""
    kv, _ = read_golden("weighting_examples.txt")
    S = num(kv["seed_example.scale"])
    counts = [int(c) for c in kv["seed_example.counts"].split()]
    seeds = [float(x) for x in kv["seed_example.seeds"].split()]
    N = sum(counts)
    for n, seed in zip(counts, seeds):
        w = lib.tlo_microbatch_weight(n, N)
        assert np.float32(S) * np.float32(w) == np.float32(seed), (n, w, seed)
        assert S * (n / N) == seed  # the page's f64 value is n/N in f64 times S


def pin_accumulation_equals_one_big_batch(lib):
    """[MP] section 4 catalogue (test_accumulation_equals_one_big_batch): micro-batches of
    5, 11 and 16 rows equal one batch of 32 rows to 1e-6.  Each micro-batch gradient is the
    gradient of that micro-batch's mean loss, i.e. the mean of its rows' gradients."""
    rng = np.random.default_rng(39)
    rows = rng.standard_normal((32, 257))
    full = rows.mean(axis=0)  # the one-batch gradient, fp64
    for sizes in ((5, 11, 16), (16, 5, 11), (1, 31), (32,)):
        bounds = np.cumsum((0,) + sizes)
        grads = [rows[a:b].mean(axis=0).astype(np.float32) for a, b in zip(bounds[:-1], bounds[1:])]
        u, res = accumulated_u(lib, grads, list(sizes))
        assert not res.skipped
        err = np.max(np.abs(u.astype(np.float64) - full))
        assert err <= 1e-6, (sizes, err)


# --------------------------------------------------------------------------
# Loss scaling: unscale, overflow flag, fp16 rescue
# --------------------------------------------------------------------------

def pin_unscale_is_exact_for_powers_of_two(lib):
    """[MP] section 2 "Loss scaling": with S a power of two, unscaling only changes the
    exponent, so u = acc * 2^-e exactly (closed form: numpy.ldexp)."""
    rng = np.random.default_rng(7)
    mant = rng.uniform(1.0, 2.0, 4096)
    expo = rng.integers(-90, 90, 4096)
    base = np.ldexp(mant, expo).astype(np.float32) * rng.choice([-1, 1], 4096).astype(np.float32)
    for e in (0, 1, 7, 10, 14, 16, 24):
        acc = base.copy()
        found = lib.tlo_unscale_check(_p(acc), acc.size, float(2.0 ** e))
        assert found == 0
        assert np.array_equal(acc.view(np.uint32), np.ldexp(base, -e).astype(np.float32).view(np.uint32)), e


def pin_overflow_flag(lib):
    """[MEG] section 6 / [MP] "Dynamic scaling": any non-finite gradient flags the step."""
    for bad in (np.inf, -np.inf, np.nan):
        acc = np.ones(1000, np.float32)
        acc[617] = bad
        assert lib.tlo_unscale_check(_p(acc), acc.size, 8.0) == 1
    acc = np.full(1000, 3.0e38, np.float32)
    assert lib.tlo_unscale_check(_p(acc), acc.size, 1.0) == 0


def pin_fp16_underflow_rescued_by_scaling(lib):
    """[MP] section 2 / catalogue test_fp16_underflow_is_rescued_by_loss_scaling:
    1e-8 flushes to zero in fp16; scaled by 2^16 it survives and unscales to within
    fp16's relative precision 2^-11.  fp16 limits: 65504, 2^-14, 2^-24."""
    kv, _ = read_golden("clip_and_rescue_examples.txt")
    g = np.float32(num(kv["rescue.g"]))
    S = num(kv["rescue.scale"])
    assert lib.tlo_f32_to_f16(float(g)) == 0  # flushed
    bits = np.array([lib.tlo_f32_to_f16(float(np.float32(S) * g))], np.uint16)
    acc = np.empty(1, np.float32)
    lib.tlo_accumulate(_p(acc), _p(bits), oracle.DT_F16, 1, 1.0, 1)
    assert lib.tlo_unscale_check(_p(acc), 1, float(S)) == 0
    assert abs(acc[0] - g) <= num(kv["rescue.rel_tol"]) * g, acc[0]
    kv2, _ = read_golden("recast_examples.txt")
    assert lib.tlo_f16_to_f32(0x7BFF) == num(kv2["fp16.max_finite"])
    assert lib.tlo_f16_to_f32(0x0400) == num(kv2["fp16.min_normal"])
    assert lib.tlo_f16_to_f32(0x0001) == num(kv2["fp16.min_subnormal"])


# --------------------------------------------------------------------------
# The dynamic loss scaler
# --------------------------------------------------------------------------

def pin_loss_scaler_five_step_trace(lib):
    """[MP] section 3 Loss scaling table (S=8, growth 2, backoff 1/2, interval 2, SGD eta 0.5):
    w = -0.5, -0.5, -1.0, -2.0, -3.0; S = 8, 4, 4, 8, 8; count = 1, 0, 1, 0, 1.
    SGD (w <- w - eta*g) is a test helper here, not part of the oracle."""
    kv, rows = read_golden("loss_scaler_trace.txt")
    st = oracle.State(num(kv["init.S"]), 0, 0, 1.0, 1.0)
    cfg = oracle.ScalerCfg(1, num(kv["growth"]), num(kv["backoff"]), int(kv["interval"]), 1.0, 2.0 ** 127)
    w = np.float32(num(kv["init.w"]))
    eta = np.float32(num(kv["eta"]))
    for step, g, w_after, S_after, count_after in rows:
        acc = np.array([num(g)], np.float32)
        found = lib.tlo_unscale_check(_p(acc), 1, st.S)
        if not found:
            w = np.float32(w - np.float32(eta * acc[0]))
        lib.tlo_scaler_update(ctypes.byref(st), ctypes.byref(cfg), found, 1.0, 1.0)
        assert w == np.float32(num(w_after)), (step, w)
        assert st.S == num(S_after), (step, st.S)
        assert st.count == int(count_after), (step, st.count)
    assert st.t == 4


def pin_rust_scaler_fixture(lib):
    """[RST] ch. 13: a commit at interval 1 takes S 128 -> 256 (optimizer step 1); an
    overflowing attempt takes S 128 -> 64 and keeps optimizer step 1."""
    kv, _ = read_golden("rust_scaler_fixture.txt")
    cfg = oracle.ScalerCfg(1, 2.0, 0.5, int(kv["commit.interval"]), 1.0, 2.0 ** 127)
    st = oracle.State(num(kv["commit.S_before"]), 0, 0, 1.0, 1.0)
    lib.tlo_scaler_update(ctypes.byref(st), ctypes.byref(cfg), 0, 0.9, 0.95)
    assert st.S == num(kv["commit.S_after"]) and st.t == int(kv["commit.t_after"])
    st = oracle.State(num(kv["overflow.S_before"]), 0, int(kv["overflow.t_before"]), 0.9, 0.95)
    lib.tlo_scaler_update(ctypes.byref(st), ctypes.byref(cfg), 1, 0.81, 0.9025)
    assert st.S == num(kv["overflow.S_after"]) and st.t == int(kv["overflow.t_after"])
    assert st.b1p == 0.9 and st.b2p == 0.95  # beta powers preserved on a skip


def pin_scaler_floor_and_cap(lib):
    """[MEG] section 5 controller: after an overflow S becomes max(S * backoff, min_loss_scale),
    so repeated overflows stop at the floor; reading R2 caps growth at max_scale."""
    cfg = oracle.ScalerCfg(1, 2.0, 0.5, 1, 4.0, 64.0)
    st = oracle.State(8.0, 0, 0, 1.0, 1.0)
    for want in (4.0, 4.0, 4.0):
        lib.tlo_scaler_update(ctypes.byref(st), ctypes.byref(cfg), 1, 1.0, 1.0)
        assert st.S == want
    for want in (8.0, 16.0, 32.0, 64.0, 64.0):
        lib.tlo_scaler_update(ctypes.byref(st), ctypes.byref(cfg), 0, 1.0, 1.0)
        assert st.S == want and st.count == 0


def fp16_scaled(g: np.ndarray, S: float) -> np.ndarray:
    """fp16 bits of S*g: what a backward pass seeded with S*L would hand over."""
    return (g.astype(np.float32) * np.float32(S)).astype(np.float16).view(np.uint16)


def pin_fp16_scale_sequence_20_steps(lib):
    """The S sequence of the 20-step fp16 workload, hand-derived from the controller rules
    ([MP] "Dynamic scaling"; [MEG] section 5): skips at 3 and 11, 18 commits, final count 1."""
    _, rows = read_golden("config1_scale_sequence.txt")
    kv, _ = read_golden("config1_scale_sequence.txt")
    rng = np.random.default_rng(39)
    P = 2048
    master = (rng.standard_normal(P) * 0.02).astype(np.float32)
    o = make_oracle(lib, master, pdtype="f16", gdtype="f16", scaler_enabled=True,
                    init_scale=2.0 ** 16, interval=4)
    for step, log2s, skipped, count in rows:
        step = int(step)
        g = rng.standard_normal(P) * 1e-6
        bits = fp16_scaled(g, o.state.S)
        if step == 3:
            bits[123] = 0x7C00
        if step == 11:
            bits[1999] = 0x7E00
        res = o.step([bits], [4096], max_norm=1.0)
        assert o.state.S == 2.0 ** int(log2s), (step, o.state.S)
        assert res.skipped == int(skipped), step
        assert o.state.count == int(count), step
    assert o.state.t == int(kv["final.t"])


def pin_skip_changes_nothing_and_drops_bad_grads(lib):
    """[RST] ch. 13 "Discard a failed partial logical update": a skipped attempt keeps weight
    bits, moments, beta powers and the optimizer step; [MP] pitfalls 12-13: a step on
    non-finite gradients or a later step that keeps them poisons the weights.  A run with a
    skipped update in the middle must equal, bit for bit, the run without it."""
    rng = np.random.default_rng(11)
    P = 777
    master = (rng.standard_normal(P) * 0.02).astype(np.float32)
    # gradients that are exact in fp16 at both scales, so unscaled values agree
    g1 = (rng.integers(-512, 512, P) * 2.0 ** -20)
    g2 = (rng.integers(-512, 512, P) * 2.0 ** -20)
    a = make_oracle(lib, master, pdtype="f16", gdtype="f16", scaler_enabled=True, init_scale=2.0 ** 10, interval=100)
    b = make_oracle(lib, master, pdtype="f16", gdtype="f16", scaler_enabled=True, init_scale=2.0 ** 10, interval=100)
    for o in (a, b):
        o.step([fp16_scaled(g1, o.state.S), fp16_scaled(g1, o.state.S)], [3, 5], max_norm=1.0)
    snap = [x.copy() for x in (a.w, a.m, a.v, a.p)] + [a.state.t, a.state.b1p, a.state.b2p]
    bad = fp16_scaled(g2, a.state.S)
    bad[5] = 0x7C00
    res = a.step([bad, fp16_scaled(g2, a.state.S)], [3, 5], max_norm=1.0)
    assert res.skipped == 1
    for before, after in zip(snap[:4], (a.w, a.m, a.v, a.p)):
        assert np.array_equal(before, after)
    assert (a.state.t, a.state.b1p, a.state.b2p) == tuple(snap[4:])
    assert a.state.S == 2.0 ** 9
    for o in (a, b):
        o.step([fp16_scaled(g2, o.state.S), fp16_scaled(g2, o.state.S)], [3, 5], max_norm=1.0)
    for x, y in ((a.w, b.w), (a.m, b.m), (a.v, b.v), (a.p, b.p)):
        assert np.array_equal(x, y)
    assert np.all(np.isfinite(a.w)) and a.state.t == b.state.t == 2


def pin_schedule_follows_committed_steps(lib):
    """[RST] ch. 13 "Discard a failed partial logical update": after one commit and one
    skipped attempt the optimizer step is still 1, and scheduled step 2 is the one still
    available.  With zero gradients only the decoupled decay acts, so the rate each update
    used can be read off exactly.  Start from w0 = 1 with weight decay 1 and rates 1/2, 1/4,
    1/8 for steps 1-3:
    - step 1 gives w = 1/2, and the skipped attempt leaves it there;
    - scheduled step 2 then gives 1/2 - 1/4 * 1/2 = 3/8 (7/16 would mean the attempt had
      consumed a step);
    - step 3 gives 21/64;
    - past the end of the table the last rate holds: 147/512."""
    table = np.array([0.5, 0.25, 0.125], np.float32)
    o = make_oracle(lib, np.ones(4, np.float32), pdtype="f16", gdtype="f32")
    zero = np.zeros(4, np.float32)
    bad = zero.copy()
    bad[1] = np.inf
    hp = dict(max_norm=0.0, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=1.0, lr_schedule=table)
    want = []
    for g in (zero, bad, zero, zero, zero):
        o.step([g], [1], **hp)
        want.append((float(o.w[0]), int(o.state.t), int(o.last.skipped)))
    assert want == [(0.5, 1, 0), (0.5, 1, 1), (0.375, 2, 0), (21 / 64, 3, 0), (147 / 512, 4, 0)], want
    assert np.all(o.w == o.w[0])


# --------------------------------------------------------------------------
# Global norm and clipping
# --------------------------------------------------------------------------

def pin_norm_brute_force_and_permutation(lib):
    """[MEG] section 9: global_norm = sqrt(sum ||g||^2).  Brute force with exact rational
    squares (math.fsum) bounds the oracle's fp32-square/fp64-sum result; the norm does not
    depend on the order of the tensors."""
    rng = np.random.default_rng(3)
    for P in (1, 7, 1000, 4099):
        u = (rng.standard_normal(P) * rng.choice([1e-3, 1.0, 30.0])).astype(np.float32)
        exact = math.fsum(float(x) * float(x) for x in u)
        s = lib.tlo_sumsq(_p(u), P)
        assert abs(s - exact) <= 2 * F32_EPS * exact, (P, s, exact)
        perm = np.ascontiguousarray(u[rng.permutation(P)])
        n1 = lib.tlo_norm_from_sumsq(s)
        n2 = lib.tlo_norm_from_sumsq(lib.tlo_sumsq(_p(perm), P))
        assert abs(n1 - n2) <= ulp32(n1)
        assert abs(n1 - math.sqrt(exact)) <= 2 * ulp32(n1)
    # a finite element whose fp32 square overflows makes the sum non-finite, and the
    # update is then skipped like an overflow (reading R4)
    u = np.array([1.0, 2.0 ** 70], np.float32)
    assert math.isinf(lib.tlo_sumsq(_p(u), 2))
    o = make_oracle(lib, np.ones(2, np.float32), gdtype="f32")
    res = o.step([u], [1], max_norm=1.0)
    assert res.skipped == 1 and o.state.t == 0 and np.all(o.w == 1.0)


def pin_clip_after_unscale_example(lib):
    """[MP] catalogue test_scaler_unscales_before_clipping: a gradient of norm 5 scaled by
    1024 clips to norm 1; [MEG] section 9: clipping before unscale would make the threshold
    depend on the loss scale."""
    kv, _ = read_golden("clip_and_rescue_examples.txt")
    u = np.array([num(x) for x in kv["clip.unscaled"].split()], np.float32)
    S = num(kv["clip.scale"])
    o = make_oracle(lib, np.zeros(2, np.float32), pdtype="f16", gdtype="f16", scaler_enabled=True,
                    init_scale=S, interval=1000)
    res = o.step([fp16_scaled(u, S)], [1], max_norm=num(kv["clip.max_norm"]))
    assert res.skipped == 0
    assert res.norm == num(kv["clip.norm"]), res.norm
    clipped = np.float32(u * np.float32(res.coef))
    assert abs(float(np.linalg.norm(clipped.astype(np.float64))) - num(kv["clip.clipped_norm"])) <= 1e-6
    # the optimizer sees the clipped gradient: from m = v = 0, m_1 = (1 - beta1) g_clipped and
    # v_1 = (1 - beta2) g_clipped^2
    gc = u.astype(np.float64) * float(np.float32(res.coef))
    assert np.allclose(o.m, (1 - float(np.float32(0.9))) * gc, rtol=4 * F32_EPS, atol=0)
    assert np.allclose(o.v, (1 - float(np.float32(0.95))) * gc * gc, rtol=8 * F32_EPS, atol=0)
    # no clipping when the norm is already within the bound
    o2 = make_oracle(lib, np.zeros(2, np.float32), pdtype="f16", gdtype="f16", scaler_enabled=True,
                     init_scale=S, interval=1000)
    res2 = o2.step([fp16_scaled(u, S)], [1], max_norm=10.0)
    assert res2.coef == 1.0


def pin_clip_matches_torch(lib):
    """Library pin: torch.nn.utils.clip_grad_norm_ (eps 1e-6, coefficient clamped at 1) in
    fp64 gives the same norm and clipped gradient as the oracle."""
    import torch
    rng = np.random.default_rng(5)
    for scale, max_norm in ((1e-2, 1.0), (1.0, 100.0), (3.0, 0.5)):
        parts = [(rng.standard_normal(n) * scale).astype(np.float32) for n in (10, 300, 77)]
        u = np.concatenate(parts)
        norm = lib.tlo_norm_from_sumsq(lib.tlo_sumsq(_p(u), u.size))
        coef = lib.tlo_clip_coef(norm, max_norm)
        ps = [torch.nn.Parameter(torch.from_numpy(x.astype(np.float64))) for x in parts]
        for p, x in zip(ps, parts):
            p.grad = torch.from_numpy(x.astype(np.float64)).clone()
        tn = float(torch.nn.utils.clip_grad_norm_(ps, max_norm))
        assert abs(norm - tn) <= 2e-7 * tn
        got = u.astype(np.float64) * coef
        want = torch.cat([p.grad for p in ps]).numpy()
        assert np.allclose(got, want, rtol=1e-6, atol=0), (scale, max_norm)
    assert lib.tlo_clip_coef(5.0, 0.0) == 1.0  # max_norm <= 0 disables clipping


# --------------------------------------------------------------------------
# AdamW on fp32 masters
# --------------------------------------------------------------------------

def _adam_run(lib, master, grads_seq, hp, max_norm=0.0):
    o = make_oracle(lib, master, pdtype="bf16", gdtype="f32")
    for g in grads_seq:
        res = o.step([np.asarray(g, np.float32)], [1], max_norm=max_norm, **hp)
        assert res.skipped == 0
    return o


def pin_adamw_first_step_closed_form(lib):
    """[ZRO] "Why the optimizer state...": the update divides the bias-corrected first moment
    by the root of the bias-corrected second moment plus a small constant.  From m = v = 0,
    after one step m_hat = g and v_hat = g^2 exactly, so (closed form, decoupled decay)
    w1 = w0 (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(1)
    w0 = (rng.standard_normal(500) * 0.5).astype(np.float32)
    g = (rng.standard_normal(500) * rng.choice([1e-6, 1e-3, 1.0], 500)).astype(np.float32)
    for hp in (dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1),
               dict(lr=3e-2, beta1=0.8, beta2=0.9, eps=1e-3, weight_decay=0.5)):
        o = _adam_run(lib, w0, [g], hp)
        w0d, gd = w0.astype(np.float64), g.astype(np.float64)
        lr, wd, eps = float(np.float32(hp["lr"])), float(np.float32(hp["weight_decay"])), float(np.float32(hp["eps"]))
        want = w0d * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
        tol = 8 * F32_EPS * (np.abs(w0d) + lr)
        assert np.all(np.abs(o.w - want) <= tol), np.max(np.abs(o.w - want) / tol)
        b1, b2 = np.float32(hp["beta1"]), np.float32(hp["beta2"])
        assert np.allclose(o.m, (1 - b1.astype(np.float64)) * gd, rtol=4 * F32_EPS, atol=0)
        assert np.allclose(o.v, (1 - b2.astype(np.float64)) * gd * gd, rtol=8 * F32_EPS, atol=0)


def pin_adamw_constant_gradient_closed_form(lib):
    """For a constant gradient g from m = v = 0, m_hat_t = g and v_hat_t = g^2 at every t, so
    with wd = 0 each step moves w by exactly lr g / (|g| + eps): w_T = w0 - T lr g/(|g|+eps).
    This fixes the bias corrections and the beta powers at every step, not only the first."""
    rng = np.random.default_rng(2)
    w0 = (rng.standard_normal(64) * 0.1).astype(np.float32)
    g = (rng.standard_normal(64) * 1e-2).astype(np.float32)
    T = 40
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)
    o = _adam_run(lib, w0, [g] * T, hp)
    gd = g.astype(np.float64)
    want = w0.astype(np.float64) - T * float(np.float32(1e-3)) * gd / (np.abs(gd) + float(np.float32(1e-8)))
    tol = 16 * T * F32_EPS * (np.abs(want) + 1e-3)
    assert np.all(np.abs(o.w - want) <= tol), np.max(np.abs(o.w - want) / tol)
    assert o.state.t == T
    assert abs(o.state.b1p - float(np.float32(0.9)) ** T) <= 1e-12


def pin_adamw_pure_decay(lib):
    """With g = 0 the moments stay 0 and only the decoupled decay acts: w_T = w0 (1 - lr wd)^T."""
    w0 = np.linspace(-1, 1, 33).astype(np.float32)
    T = 25
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.3)
    o = _adam_run(lib, w0, [np.zeros(33, np.float32)] * T, hp)
    lrwd = float(np.float32(float(np.float32(1e-2)) * float(np.float32(0.3))))
    want = w0.astype(np.float64) * (1 - lrwd) ** T
    assert np.all(np.abs(o.w - want) <= 4 * T * F32_EPS * np.abs(w0) + 1e-30)
    assert np.all(o.m == 0) and np.all(o.v == 0)


def pin_adamw_matches_torch(lib):
    """Library pin: torch.optim.AdamW (decoupled decay, eps outside the root) in fp64 over
    many steps, with plain and exaggerated hyper-parameters so that every term of the
    update (each bias correction, eps, decay, each beta) moves the result well beyond
    fp32 rounding."""
    import torch
    rng = np.random.default_rng(4)
    P, T = 300, 30
    w0 = (rng.standard_normal(P) * 0.05).astype(np.float32)
    gs = [(rng.standard_normal(P) * 1e-2 * (1 + (t % 3))).astype(np.float32) for t in range(T)]
    for hp in (dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1),
               dict(lr=2e-2, beta1=0.7, beta2=0.8, eps=3e-3, weight_decay=0.9)):
        o = _adam_run(lib, w0, gs, hp)
        f = {k: float(np.float32(v)) for k, v in hp.items()}
        p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
        opt = torch.optim.AdamW([p], lr=f["lr"], betas=(f["beta1"], f["beta2"]), eps=f["eps"],
                                weight_decay=f["weight_decay"])
        for g in gs:
            p.grad = torch.from_numpy(g.astype(np.float64))
            opt.step()
        st = opt.state[p]
        want_w = p.detach().numpy()
        scale_w = np.abs(want_w) + f["lr"] * T
        assert np.all(np.abs(o.w - want_w) <= 8 * T * F32_EPS * scale_w), np.max(np.abs(o.w - want_w) / scale_w)
        assert np.allclose(o.m, st["exp_avg"].numpy(), rtol=0, atol=64 * F32_EPS * np.max(np.abs(o.m)))
        assert np.allclose(o.v, st["exp_avg_sq"].numpy(), rtol=0, atol=64 * F32_EPS * np.max(np.abs(o.v)))


# --------------------------------------------------------------------------
# Recast and 16-bit formats
# --------------------------------------------------------------------------

def pin_recast_worked_examples(lib):
    """[MP] section 3: 1 + 2^-8 -> bf16 1.0 (tie to even); 1.01 -> 1.0078125."""
    kv, _ = read_golden("recast_examples.txt")
    for key in ("tie", "near"):
        bits = lib.tlo_f32_to_bf16(float(np.float32(num(kv[key + ".input"]))))
        assert lib.tlo_bf16_to_f32(bits) == num(kv[key + ".bf16"]), key


def pin_master_keeps_sub_bf16_update(lib):
    """[MP] section 2 "Why the weights stay float32": a weight of 1 moved by 1e-3 stays 1.0 in
    bf16 but the fp32 master moves; repeated small updates then reach the bf16 copy."""
    kv, _ = read_golden("recast_examples.txt")
    w0 = np.array([num(kv["master.init"])], np.float32)
    hp = dict(lr=num(kv["master.update"]), beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)
    o = _adam_run(lib, w0, [np.ones(1, np.float32)], hp)
    assert o.w[0] != 1.0 and abs(o.w[0] - (1 - 1e-3)) < 1e-6
    assert lib.tlo_bf16_to_f32(int(o.p[0])) == num(kv["master.bf16_after"])
    o = _adam_run(lib, w0, [np.ones(1, np.float32)] * 3, hp)
    assert lib.tlo_bf16_to_f32(int(o.p[0])) == 1.0 - 2.0 ** -8  # nearest bf16 to 0.997


def pin_conversions_match_libraries(lib):
    """Library pin: every 16-bit pattern decodes as numpy float16 / torch bfloat16 do, and fp32
    values at and around every rounding boundary encode as they round (RNE)."""
    import torch
    allbits = np.arange(65536, dtype=np.uint16)
    dec16 = np.empty(65536, np.float32)
    lib.tlo_decode16(_p(allbits), _p(dec16), 65536, oracle.DT_F16)
    want16 = allbits.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(dec16), np.isnan(want16))
    ok = ~np.isnan(want16)
    assert np.array_equal(dec16[ok].view(np.uint32), want16[ok].view(np.uint32))
    decb = np.empty(65536, np.float32)
    lib.tlo_decode16(_p(allbits), _p(decb), 65536, oracle.DT_BF16)
    wantb = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).float().numpy()
    ok = ~np.isnan(wantb)
    assert np.array_equal(decb[ok].view(np.uint32), wantb[ok].view(np.uint32))
    # encode: neighbours of all finite 16-bit values, the midpoints and +-1 fp32 ulp around them
    rng = np.random.default_rng(9)
    for fmt in ("f16", "bf16"):
        vals = (dec16 if fmt == "f16" else decb)
        fin = np.sort(np.unique(vals[np.isfinite(vals)]).astype(np.float64))
        mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)
        cand = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf)),
                               fin.astype(np.float32),
                               rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
                               np.array([np.inf, -np.inf, 65504, 65519.99, 65520, 1e-8, 2 ** -25, 3 * 2 ** -26,
                                         2 ** -149, 3.4e38], np.float32)])
        cand = cand[~np.isnan(cand)].astype(np.float32)
        out = np.empty(cand.size, np.uint16)
        lib.tlo_recast(_p(cand), _p(out), cand.size, oracle.dtype_code(fmt))
        if fmt == "f16":
            with np.errstate(over="ignore"):
                want = cand.astype(np.float16).view(np.uint16)
        else:
            want = torch.from_numpy(cand).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        bad = np.nonzero(out != want)[0]
        assert bad.size == 0, (fmt, cand[bad[:5]], out[bad[:5]], want[bad[:5]])
    # NaN stays NaN in both formats
    assert np.isnan(lib.tlo_f16_to_f32(lib.tlo_f32_to_f16(float("nan"))))
    assert np.isnan(lib.tlo_bf16_to_f32(lib.tlo_f32_to_bf16(float("nan"))))


def pin_state_bytes_per_param(lib):
    """[T41] eq. (41.1), [MEG] section 1: 2 + 2 + 4 + 4 + 4 = 16 bytes per parameter of model
    state (plus 4 for the fp32 accumulation buffer)."""
    kv, _ = read_golden("memory_accounting.txt")
    o = make_oracle(lib, np.zeros(10, np.float32), pdtype="bf16", gdtype="bf16")
    grad_itemsize = 2  # a bf16/fp16 gradient
    parts = {"model_param": o.p.itemsize, "model_grad": grad_itemsize, "master": o.w.itemsize,
             "adam_m": o.m.itemsize, "adam_v": o.v.itemsize}
    for k, v in parts.items():
        assert v == int(kv[k]), k
    assert sum(parts.values()) == int(kv["total"])
    assert sum(parts.values()) + o.acc.itemsize == 20


def pin_nonfinite_without_scaler_still_skips(lib):
    """[MP] "Dynamic scaling": bf16 needs no scaler, but a finite check still gates the
    step (pitfall s17: stepping on a NaN when the scaler is off).  With the scaler
    disabled a NaN or inf gradient skips the update: weights, moments, model copy, t and
    S = 1 unchanged; the next clean update commits as usual."""
    rng = np.random.default_rng(17)
    master = rng.standard_normal(64).astype(np.float32) * 0.02
    o = make_oracle(lib, master, pdtype="bf16", gdtype="f32")
    g = [rng.standard_normal(64).astype(np.float32) * 1e-2 for _ in range(2)]
    o.step(g, [2, 3], 1.0)
    before = [x.copy() for x in (o.w, o.m, o.v, o.p)]
    t0 = o.state.t
    for bad in (np.nan, np.inf):
        gb = [x.copy() for x in g]
        gb[1][7] = bad
        r = o.step(gb, [2, 3], 1.0)
        assert r.skipped == 1 and o.state.t == t0 and o.state.S == 1.0 and o.state.count == 0
        for a, b in zip(before, (o.w, o.m, o.v, o.p)):
            assert np.array_equal(a, b)
    r = o.step(g, [2, 3], 1.0)
    assert r.skipped == 0 and o.state.t == t0 + 1


def pin_resume_keeps_the_good_step_count(lib):
    """[MP] section 4: the scaler's state_dict keeps S and the good-step count (pitfall
    s16: losing the count on resume).  An update sequence interrupted after 3 steps and
    resumed from (S, count, t, beta powers, w, m, v, param) ends exactly where the
    uninterrupted one does, S growing at the same step (interval 4)."""
    rng = np.random.default_rng(16)
    master = rng.standard_normal(32).astype(np.float32) * 0.02
    grads = [[fp16_scaled(rng.standard_normal(32).astype(np.float32) * 1e-3, 2.0 ** 8)] for _ in range(7)]
    kw = dict(pdtype="f16", gdtype="f16", scaler_enabled=True, init_scale=2.0 ** 8, interval=4)
    a = make_oracle(lib, master, **kw)
    seq_a = []
    for g in grads:
        a.step(g, [5], 1.0)
        seq_a.append(a.state.S)
    b = make_oracle(lib, master, **kw)
    for g in grads[:3]:
        b.step(g, [5], 1.0)
    c = make_oracle(lib, master, **kw)
    for f in ("w", "m", "v", "p"):
        setattr(c, f, getattr(b, f).copy())
    c.state = oracle.State(b.state.S, b.state.count, b.state.t, b.state.b1p, b.state.b2p)
    assert c.state.count == 3
    seq_c = []
    for g in grads[3:]:
        c.step(g, [5], 1.0)
        seq_c.append(c.state.S)
    assert seq_c == seq_a[3:] and seq_a[3] == 2.0 ** 9 and seq_a[2] == 2.0 ** 8
    for f in ("w", "m", "v", "p"):
        assert np.array_equal(getattr(a, f), getattr(c, f)), f
    assert (a.state.S, a.state.count, a.state.t) == (c.state.S, c.state.count, c.state.t)


# ---- 8-bit gradients with fine-grained scaling ([T41] section 41.5) --------

def _torch_e4m3(codes):
    """Library decode of E4M3 codes: torch.float8_e4m3fn."""
    import torch
    return torch.tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def pin_e4m3_decode_matches_torch(lib):
    """Library pin: every one of the 256 E4M3 codes decodes as torch.float8_e4m3fn does
    (values bit for bit, signed zeros, NaN exactly at S.1111.111, no infinity)."""
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([lib.tlo_e4m3_to_f32(int(c)) for c in codes], dtype=np.float32)
    ref = _torch_e4m3(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert not np.isinf(ours).any()


def pin_e4m3_closed_forms(lib):
    """R17's layout in closed form: largest finite 1.75 * 2^8 = 448, smallest subnormal
    2^-9, smallest normal 2^-6, 0x38 = 1; the 127 non-negative finite codes increase."""
    d = lambda c: lib.tlo_e4m3_to_f32(c)
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6 and d(0x38) == 1.0 and d(0x39) == 1.125
    assert math.copysign(1.0, d(0x80)) == -1.0 and d(0x80) == 0.0
    vals = [d(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))


def _quantize_blocks(x, numel):
    """[T41] section 41.5 recipe (block 16, per-block scale max|x|/448, 1 where the block
    is zero, values coded relative to the scale), per tensor, with torch's RNE cast."""
    import torch
    codes, scales, o = [], [], 0
    for n in numel:
        t = torch.tensor(x[o:o + n], dtype=torch.float32)
        nb = (n + 15) // 16
        pad = torch.zeros(nb * 16, dtype=torch.float32)
        pad[:n] = t
        amax = pad.view(nb, 16).abs().amax(dim=1)
        sc = amax / 448.0
        sc = torch.where(sc == 0, torch.ones_like(sc), sc)
        q = (pad.view(nb, 16) / sc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1)[:n]
        codes.append(q.numpy())
        scales.append(sc.numpy())
        o += n
    return np.concatenate(codes), np.concatenate(scales).astype(np.float32)


def pin_block_dequant_roundtrip(lib):
    """[T41] section 41.5: a block's largest magnitude codes as 448 and dequantizes back to
    itself within one fp32 rounding; every value of the normal E4M3 range comes back within
    half an E4M3 step (relative 2^-4), every subnormal within 2^-10 of the block scale."""
    rng = np.random.default_rng(41)
    numel = [16, 5, 17, 33, 64]
    x = (rng.standard_normal(sum(numel)) * np.exp(rng.uniform(-6, 6, sum(numel)))).astype(np.float32)
    codes, scales = _quantize_blocks(x, numel)
    dq = oracle.dequant_e4m3b16(codes, scales, numel)
    o, b = 0, 0
    for n in numel:
        for blk in range(0, n, 16):
            xs = x[o + blk:o + min(blk + 16, n)].astype(np.float64)
            ds = dq[o + blk:o + min(blk + 16, n)].astype(np.float64)
            s = float(scales[b])
            i = int(np.argmax(np.abs(xs)))
            assert abs(ds[i] - xs[i]) <= ulp32(xs[i]), (ds[i], xs[i])
            rel = np.abs(xs) / s
            normal = rel >= 2.0 ** -6
            assert np.all(np.abs(ds - xs)[normal] <= 2.0 ** -4 * np.abs(xs)[normal] * (1 + 1e-6))
            assert np.all(np.abs(ds - xs)[~normal] <= 2.0 ** -10 * s * (1 + 1e-6))
            b += 1
        o += n


def pin_block_scales_follow_tensors(lib):
    """R18: block scales run over each tensor separately (blocks of 16, a partial last
    block per tensor): with every code 1.0 the dequantized list is each tensor's scales
    repeated 16 times and cut to its size."""
    numel = [5, 16, 17, 33, 1, 40]
    nb = [(n + 15) // 16 for n in numel]
    scales = (2.0 ** np.arange(1, sum(nb) + 1)).astype(np.float32)
    codes = np.full(sum(numel), 0x38, dtype=np.uint8)
    dq = oracle.dequant_e4m3b16(codes, scales, numel)
    expect, b = [], 0
    for n, k in zip(numel, nb):
        expect.append(np.repeat(scales[b:b + k], 16)[:n])
        b += k
    assert np.array_equal(dq, np.concatenate(expect))


def pin_e4m3_step_equals_step_on_dequantized(lib):
    """The 8-bit path is the fp32 path on the dequantized values: one update with E4M3
    gradients equals, bit for bit, the update with fp32 gradients code * scale."""
    rng = np.random.default_rng(7)
    numel = [40, 17, 3]
    P = sum(numel)
    master = rng.standard_normal(P).astype(np.float32) * 0.02
    grads = [rng.standard_normal(P).astype(np.float32) * 1e-2 for _ in range(3)]
    q = [_quantize_blocks(g, numel) for g in grads]
    a = make_oracle(lib, master, pdtype="bf16", gdtype="f32")
    b = oracle.Oracle(master, oracle.recast(master, "bf16"), param_dtype="bf16", grad_dtype="e4m3b16",
                      lib=lib, numel=numel)
    for _ in range(2):
        ra = a.step([oracle.dequant_e4m3b16(c, s, numel) for c, s in q], [3, 1, 2], 1.0)
        rb = b.step(q, [3, 1, 2], 1.0)
        assert (ra.norm, ra.sumsq, ra.skipped) == (rb.norm, rb.sumsq, rb.skipped)
    for f in ("w", "m", "v", "p"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    bad = [(c.copy(), s) for c, s in q]
    bad[1][0][20] = 0x7F                                   # a NaN code flags the update
    r = b.step(bad, [3, 1, 2], 1.0)
    assert r.skipped == 1


# --------------------------------------------------------------------------
# The sharded step ([ZRO] "The scheme", "Operational sharp edges"; [MEG] sections 6, 9)
# --------------------------------------------------------------------------

def pin_partition_covers_every_element_once(lib):
    """The slices of the sharded statement: disjoint, covering [0, P) in order, cut on
    multiples of align, and balanced (each cut within align of j*P/N), for lists shorter
    than the rank count, empty lists and uneven sizes; every element counted once by brute
    force on small cases."""
    cases = [(0, 3, 1), (5, 8, 1), (100, 3, 16), (1000, 7, 1), (1000, 7, 16), (12345, 5, 8),
             (2 ** 40 + 3, 6, 16), (16, 16, 16), (17, 2, 16)]
    for P, N, align in cases:
        b = oracle.partition_bounds(P, N, align)
        assert b[0] == 0 and b[-1] == P and b.size == N + 1, (P, N, align)
        assert np.all(np.diff(b) >= 0), (P, N, align)
        for j in range(1, N):
            assert b[j] % align == 0, (P, N, align)
            assert 0 <= Fraction(j * P, N) - b[j] < align, (P, N, align, j)
        if P <= 20000:
            owners = np.zeros(P, dtype=np.int64)
            for r in range(N):
                owners[b[r]:b[r + 1]] += 1
            assert np.all(owners == 1), (P, N, align)


def pin_sharded_step_equals_unsharded(lib):
    """[ZRO]: N devices each updating their own slice, with the squared norms all-reduced
    before the root and the overflow flag all-reduced ([MEG] section 6), compute the update
    of one device holding everything.  Per element the operations are the same, so the
    state is bit-identical whenever the fp32 norm is (it is here); the squared norm differs
    only by the fp64 association of the rank sums (equal for one rank).  An overflow in the
    last rank's slice makes every rank skip; each rank's squared norm is its slice's."""
    rng = np.random.default_rng(11)
    numel = [37, 4096, 5, 999, 2048, 1]
    P = sum(numel)
    master = rng.standard_normal(P).astype(np.float32) * 0.02
    for N, align in ((1, 1), (2, 1), (3, 16), (5, 16), (2, 64)):
        ref = make_oracle(lib, master, pdtype="f16", gdtype="f16", scaler_enabled=True, init_scale=2.0 ** 10,
                          interval=2, numel=numel)
        shd = make_oracle(lib, master, pdtype="f16", gdtype="f16", scaler_enabled=True, init_scale=2.0 ** 10,
                          interval=2, numel=numel)
        bounds = oracle.partition_bounds(P, N, align)
        for step in range(5):
            grads = [oracle.recast(rng.standard_normal(P).astype(np.float32) * 0.05 * ref.state.S, "f16")
                     for _ in range(3)]
            if step == 3:
                grads[1][P - 2] = 0x7C00               # +inf in the last slice only
            ra = ref.step(grads, [3, 1, 2], 1.0)
            rb = shd.step(grads, [3, 1, 2], 1.0, shards=(N, align))
            assert (ra.skipped, ra.found_inf) == (rb.skipped, rb.found_inf) == ((1, 1) if step == 3 else (0, 0))
            assert shd.rank_flag[-1] == (1 if step == 3 else 0) and not np.any(shd.rank_flag[:-1])
            if not ra.skipped:
                assert ra.norm == rb.norm and ra.coef == rb.coef and ra.coef < 1.0
                assert abs(ra.sumsq - rb.sumsq) <= 1e-12 * ra.sumsq
                if N == 1:
                    assert ra.sumsq == rb.sumsq
                for r in range(N):   # each rank's squared norm is its own slice's
                    assert shd.rank_sumsq[r] == lib.tlo_sumsq(
                        shd.acc[bounds[r]:].ctypes.data_as(ctypes.c_void_p), int(bounds[r + 1] - bounds[r]))
            assert ref.scalars() == shd.scalars()
            for f in ("w", "m", "v", "p"):
                assert np.array_equal(getattr(ref, f), getattr(shd, f)), (N, align, step, f)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
