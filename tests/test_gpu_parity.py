"""GPU parity: the CUDA library (through its C ABI) against the oracle on the same
seeded inputs.

Tolerances (fixed by the method's statement of what must agree):
  overflow flags, skip decisions, the loss-scale sequence, the good-step count, t and
  the beta powers: bit-exact;
  fp32 master, m, v: at most 2 units in the last place per element;
  bf16/fp16 parameters: at most 1 unit in the last place;
  the global gradient norm: 1e-6 relative.
"""
import ctypes
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W
from harness import (DT, GpuOptimizer, assert_ulps16, assert_ulps32, compare_scalars, compare_state,
                     grad_bits, oracle_for, run_parity)
from oracle_pins import read_golden

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def custom(numel, pdtype="bf16", gdtype="bf16", k=2, steps=2, scaler=False, init_scale=1.0, interval=2000,
           grad_std=1e-2, counts=None, injections=None, name="custom"):
    return W.Workload(name, list(numel), pdtype, gdtype, steps=steps, k=k, grad_std=grad_std, scaler_enabled=scaler,
                      init_scale=init_scale, interval=interval, fixed_counts=counts,
                      grads_prescaled=scaler, injections=injections or {})


# ---------------------------------------------------------------------------
# the workloads at their stated sizes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gaps", [False, True], ids=["aligned", "misaligned"])
def test_bf16_small(gaps):
    """12 x 4,096 bf16, k=2 with 6 and 3 targets, clip active, 3 steps."""
    _, _, log = run_parity(W.make("bf16_small"), gaps=gaps)
    assert all(e["norm_oracle"] > 1.0 for e in log)  # the clip is active


def test_fp16_scaled_sequence():
    """64 x 16,384 fp16 with dynamic loss scaling over 20 steps: skips at 3 and 11 and the
    hand-derived S sequence, on the GPU."""
    _, rows = read_golden("config1_scale_sequence.txt")
    gpu, orc, log = run_parity(W.make("fp16_scaled"), compare_every=5)
    for e, (step, log2s, skipped, count) in zip(log, rows):
        assert e["S"] == 2.0 ** int(log2s) and e["skipped"] == int(skipped), e
    assert gpu.status().t == 18


def test_llama_10m():
    """The ~10.3M-parameter Llama tensor list, k=4 with 5-20% padding, 10 steps."""
    run_parity(W.make("llama_10m"), compare_every=5)


# ---------------------------------------------------------------------------
# hyper-parameters, clipping off, and the loss scale's floor and cap
# ---------------------------------------------------------------------------

# A second common setting (betas 0.9 / 0.999, eps 1e-6, no weight decay) and an
# exaggerated one (small betas, a large eps and decay), so that a slip in the bias
# corrections, the eps placement or the decay shows at the parity tolerances.
HP_SETS = {
    "adam_0999": dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-6, weight_decay=0.0),
    "exaggerated": dict(lr=1e-3, beta1=0.7, beta2=0.8, eps=3e-3, weight_decay=0.9),
}


@pytest.mark.parametrize("hp", list(HP_SETS), ids=list(HP_SETS))
@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
def test_hyper_parameter_sets(hp, resident):
    """The kernels' AdamW constants and element update under two more hyper-parameter sets,
    6 updates from zero moments, ragged misaligned tensors, clip active."""
    wl = custom([5000, 300, 20000, 17, 2 * 16384 + 5, 1], k=3, steps=6, counts=[3, 4, 2], grad_std=3e-2)
    _, _, log = run_parity(wl, gaps=True, hp=HP_SETS[hp], resident=resident)
    assert all(e["norm_oracle"] > 1.0 for e in log)


@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
def test_clip_disabled(resident):
    """max_norm = 0 disables clipping ([MEG] section 9 clip, read as off for max_norm <= 0):
    coefficient 1 although the norm (about 1.65) is above 1."""
    gpu, orc, log = run_parity(W.make("bf16_small"), max_norm=0.0, resident=resident)
    st = gpu.status()
    assert st.coef == 1.0 and all(e["norm_oracle"] > 1.0 for e in log)


def test_scaler_floor_and_cap():
    """[MEG] section 5: the scale never backs off below min_loss_scale, and (reading R2) never
    grows past max_scale.  fp16, S0 = 2^16, growth every 2 clean updates, cap 2^17, floor
    2^14; updates 5-9 overflow.  S after each update, derived by hand from the rules:
    2^16, 2^17 (grown), 2^17, 2^17 (capped), 2^16, 2^15, 2^14, 2^14 (floored), 2^14,
    2^14, 2^15, 2^15; the GPU and the oracle agree on every one."""
    inj = {(s, 0): [(1234 + s, 0x7C00)] for s in range(5, 10)}
    wl = W.Workload("floor_cap", [5000, 300, 20000], "f16", "f16", steps=12, k=1, grad_std=1e-4,
                    scaler_enabled=True, init_scale=2.0 ** 16, interval=2, min_scale=2.0 ** 14,
                    max_scale=2.0 ** 17, fixed_counts=[64], grads_prescaled=True, injections=inj)
    gpu, orc, log = run_parity(wl, gaps=True, compare_every=3)
    expect = [16, 17, 17, 17, 16, 15, 14, 14, 14, 14, 15, 15]
    assert [e["S"] for e in log] == [2.0 ** x for x in expect]
    assert [e["skipped"] for e in log] == [0] * 4 + [1] * 5 + [0] * 3
    assert gpu.status().t == 7


# ---------------------------------------------------------------------------
# ragged, misaligned, empty and degenerate lists
# ---------------------------------------------------------------------------

EDGE_LISTS = {
    "one_element": [1],
    "tails": [1, 7, 9, 127, 16383, 16384, 16385, 3 * 16384 + 5, 33],
    "with_empty": [0, 5, 0, 4096, 0],
    "odd_sizes": [3, 1023, 2047, 65537],
}


@pytest.mark.parametrize("lst", list(EDGE_LISTS), ids=list(EDGE_LISTS))
@pytest.mark.parametrize("dtypes", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("f16", "bf16")],
                         ids=lambda d: f"p{d[0]}-g{d[1]}")
@pytest.mark.parametrize("gaps", [False, True, "packed"], ids=["aligned", "misaligned", "packed"])
@pytest.mark.parametrize("grouped", [False, True], ids=["ungrouped", "grouped"])
def test_edge_lists(lst, dtypes, gaps, grouped, monkeypatch):
    """grouped: every small tensor goes to the one-warp-per-tensor group part of the table
    (as on lists with many small tensors), else the few small tensors of these lists are
    whole-CTA segments of their own."""
    if grouped:
        monkeypatch.setenv("TL_SMALL_GROUP_MIN", "1")
    wl = custom(EDGE_LISTS[lst], pdtype=dtypes[0], gdtype=dtypes[1], k=3, steps=2, counts=[5, 1, 7])
    run_parity(wl, gaps=gaps)
    for resident in (True, "remat"):
        run_parity(wl, gaps=gaps, resident=resident)


@pytest.mark.parametrize("resident,launches", [(True, 2), ("remat", 2), (False, 5)],
                         ids=["resident", "remat", "per_microbatch"])
def test_launches_per_update_on_the_mid_size_list(resident, launches):
    """The ~10.3M-parameter list (few small tensors, few enough chunks that the pass
    finishes the norm itself, the scaler running at the end of the AdamW launch): the
    resident and re-materialising updates are two launches, the per-micro-batch one k + 1
    (three accumulations, the last micro-batch's pass, AdamW); the results still match the
    oracle over 2 updates."""
    wl = W.make("llama_10m")
    gpu, orc, log = run_parity(wl, steps=2, resident=resident)
    assert tl.tl_launch_count(gpu.ctx) == 2 * launches


@pytest.mark.parametrize("k", [1, 2, 5])
def test_micro_batch_counts(k):
    wl = custom([1000, 20000, 17], k=k, steps=2, counts=list(range(3, 3 + k)))
    run_parity(wl, gaps=True)


def test_empty_tensor_list():
    """No tensors at all: the update still runs, commits and advances the scalars."""
    wl = custom([], k=2, steps=3, counts=[2, 2])
    gpu = GpuOptimizer(wl, torch.zeros(0))
    for _ in range(3):
        gpu.step([torch.zeros(0, dtype=torch.bfloat16)] * 2, [2, 2])
    st = gpu.status()
    assert st.t == 3 and st.skipped == 0 and st.norm == 0.0
    assert st.b1p == float(np.float32(0.9)) ** 3 or abs(st.b1p - float(np.float32(0.9)) ** 3) < 1e-15


def test_all_accumulated_then_unscale_null():
    """tl_unscale_check(grads=NULL) after all k micro-batches went through tl_accumulate."""
    wl = custom([4096, 333, 70000], k=3, steps=1, counts=[4, 4, 1])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0, gaps=True)
    orc = oracle_for(wl, master0)
    grads = [W.grad_input(wl, 1, i) for i in range(3)]
    ptrs = [gpu.grad_list(i, g) for i, g in enumerate(grads)]
    for i in range(3):
        tl.tl_accumulate(gpu.ctx, ptrs[i], [4, 4, 1][i], 9, 1 if i == 0 else 0)
    tl.tl_unscale_check(gpu.ctx, None, 0, 9)
    tl.tl_grad_norm(gpu.ctx, 1.0)
    tl.tl_clip_adamw_step(gpu.ctx, tl.tl_adamw_hp(**W.HP))
    tl.tl_scaler_update(gpu.ctx)
    res = orc.step([grad_bits(g) for g in grads], [4, 4, 1], 1.0, **W.HP)
    compare_scalars(gpu.status(), orc, res, "null-grads path")
    compare_state(gpu.pull(), orc, wl, "null-grads path")


@pytest.mark.parametrize("ntensors", [512, 513, 700])
def test_long_lists_and_pointer_table_cache(ntensors):
    """Lists longer than the by-value limit use cached device pointer tables; 20 distinct
    gradient lists (more than the cache holds) force evictions."""
    rng = np.random.default_rng(ntensors)
    numel = [int(x) for x in rng.integers(1, 300, ntensors)]
    wl = custom(numel, k=2, steps=10, counts=[3, 5])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0, gaps=True)
    orc = oracle_for(wl, master0)
    for step in range(1, 11):
        grads = [W.grad_input(wl, step, i) for i in range(2)]
        slots = [(2 * step + i) % 20 for i in range(2)]
        mbs = [gpu.grad_list(s, g) for s, g in zip(slots, grads)]
        tl.logical_update(gpu.ctx, mbs, [3, 5], 1.0, tl.tl_adamw_hp(**W.HP))
        res = orc.step([grad_bits(g) for g in grads], [3, 5], 1.0, **W.HP)
        compare_scalars(gpu.status(), orc, res, f"long list step {step}")
    compare_state(gpu.pull(), orc, wl, "long list")


# ---------------------------------------------------------------------------
# skip semantics, order of calls, state round trip, graphs, determinism
# ---------------------------------------------------------------------------

def test_skip_leaves_state_bitwise_unchanged():
    """An overflowing update leaves master, m, v, params, t and beta powers bit-identical and
    halves S; the next update carries nothing of the bad gradients."""
    wl = custom([5000, 12345], pdtype="f16", gdtype="f16", k=2, steps=3, scaler=True, init_scale=2.0 ** 12,
                interval=100, counts=[2, 7], injections={(2, 1): [(17, 0x7C00)]})
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0, gaps=True)
    orc = oracle_for(wl, master0)
    before = None
    for step in (1, 2, 3):
        grads = [W.grad_input(wl, step, i, scale=orc.state.S) for i in range(2)]
        gpu.step(grads, [2, 7])
        res = orc.step([grad_bits(g) for g in grads], [2, 7], 1.0, **W.HP)
        st = gpu.status()
        compare_scalars(st, orc, res, f"skip test step {step}")
        now = gpu.pull()
        if step == 1:
            before = now
        if step == 2:
            assert st.skipped == 1 and st.S == 2.0 ** 11 and st.t == 1
            for k in ("master", "m", "v", "param"):
                assert np.array_equal(before[k].view(np.uint8), now[k].view(np.uint8)), k
    compare_state(gpu.pull(), orc, wl, "after the skip")
    assert gpu.status().t == 2


@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
def test_nonfinite_without_scaler_skips(resident):
    """bf16 without a loss scaler (the finite check still gates every update): a NaN and
    then an inf gradient skip their updates with S = 1 kept, and the state stays within
    the parity tolerances of the oracle throughout."""
    wl = custom([5000, 300, 20000], k=2, steps=4, counts=[3, 4],
                injections={(2, 0): [(123, 0x7FC0)], (3, 1): [(20100, 0x7F80)]})
    _, _, log = run_parity(wl, resident=resident)
    assert [e["skipped"] for e in log] == [0, 1, 1, 0]
    assert all(e["S"] == 1.0 for e in log)


def _small_ctx(scaler=False):
    wl = custom([100, 28], k=2, steps=1, counts=[1, 1], scaler=scaler, init_scale=8.0, interval=3,
                pdtype="f16" if scaler else "bf16", gdtype="f16" if scaler else "bf16")
    gpu = GpuOptimizer(wl, W.master_init(wl))
    g = gpu.grad_list(0, W.grad_input(wl, 1, 0, scale=8.0))
    return gpu, g


def test_call_order_and_count_errors():
    gpu, g = _small_ctx()
    ctx = gpu.ctx
    hp = tl.tl_adamw_hp(**W.HP)

    def expect(status, fn, *args):
        with pytest.raises(tl.TLError) as ei:
            fn(*args)
        assert ei.value.status == status, str(ei.value)

    expect(tl.TL_ESTATE, tl.tl_accumulate, ctx, g, 1, 2, 0)      # first=0 with nothing open
    expect(tl.TL_ESTATE, tl.tl_grad_norm, ctx, 1.0)
    expect(tl.TL_ESTATE, tl.tl_clip_adamw_step, ctx, hp)
    expect(tl.TL_ESTATE, tl.tl_scaler_update, ctx)
    expect(tl.TL_EINVAL, tl.tl_accumulate, ctx, g, 0, 2, 1)      # n_i = 0
    expect(tl.TL_EINVAL, tl.tl_accumulate, ctx, g, 3, 2, 1)      # n_i > N
    expect(tl.TL_EINVAL, tl.tl_accumulate, ctx, g, 1, 2 ** 53 + 1, 1)
    expect(tl.TL_EINVAL, tl.tl_unscale_check, ctx, g, 1, 2)      # only micro-batch must be all of N
    tl.tl_accumulate(ctx, g, 1, 3, 1)
    expect(tl.TL_EINVAL, tl.tl_accumulate, ctx, g, 1, 4, 0)      # N changed mid-update
    expect(tl.TL_EINVAL, tl.tl_unscale_check, ctx, g, 1, 3)      # 1 + 1 != 3
    expect(tl.TL_EINVAL, tl.tl_unscale_check, ctx, None, 0, 3)   # accumulated 1 != 3
    tl.tl_accumulate(ctx, g, 1, 3, 0)
    tl.tl_unscale_check(ctx, g, 1, 3)
    expect(tl.TL_ESTATE, tl.tl_unscale_check, ctx, g, 1, 3)
    expect(tl.TL_ESTATE, tl.tl_accumulate, ctx, g, 1, 3, 1)      # past accumulation
    expect(tl.TL_ESTATE, tl.tl_set_state, ctx, tl.tl_state(1.0, 0, 0, 1.0, 1.0))
    tl.tl_grad_norm(ctx, 1.0)
    expect(tl.TL_EINVAL, tl.tl_clip_adamw_step, ctx, tl.tl_adamw_hp(1e-3, 1.0, 0.95, 1e-8, 0.1))
    tl.tl_clip_adamw_step(ctx, hp)
    tl.tl_scaler_update(ctx)
    st = gpu.status()
    assert st.t == 1 and st.skipped == 0


def test_restart_discards_partial_update():
    """first=1 while an update is open restarts it: the partial sum is discarded."""
    wl = custom([3000], k=2, steps=1, counts=[1, 2])
    master0 = W.master_init(wl)
    a = GpuOptimizer(wl, master0)
    b = GpuOptimizer(wl, master0, key=50)
    junk = W.grad_input(wl, 9, 0) * 1000
    g = [W.grad_input(wl, 1, i) for i in range(2)]
    pa = [a.grad_list(i, x) for i, x in enumerate(g)]
    tl.tl_accumulate(a.ctx, a.grad_list(5, junk), 1, 3, 1)
    tl.logical_update(a.ctx, pa, [1, 2], 1.0, tl.tl_adamw_hp(**W.HP))
    b.step(g, [1, 2])
    ra, rb = a.pull(), b.pull()
    for k in ra:
        assert np.array_equal(ra[k], rb[k]), k


def test_state_roundtrip_resume():
    """[MP] section 4: a resume keeps S and the good-step count; bad arguments raise."""
    wl = custom([4096, 100], pdtype="f16", gdtype="f16", k=1, steps=7, scaler=True, init_scale=2.0 ** 10,
                interval=3, counts=[10], injections={(4, 0): [(3, 0x7C00)]})
    master0 = W.master_init(wl)
    a = GpuOptimizer(wl, master0)
    orc = oracle_for(wl, master0)
    for step in range(1, 6):
        grads = [W.grad_input(wl, step, 0, scale=orc.state.S)]
        a.step(grads, [10])
        orc.step([grad_bits(x) for x in grads], [10], 1.0, **W.HP)
    st = tl.tl_get_state(a.ctx)
    assert (st.S, st.count, st.t) == (orc.state.S, orc.state.count, orc.state.t)
    # resume into a fresh context over copies of the tensors
    b = GpuOptimizer(wl, master0, key=70)
    for name in ("master", "m", "v", "param"):
        b.lists[name].buf.copy_(a.lists[name].buf)
    tl.tl_set_state(b.ctx, st)
    for step in (6, 7):
        grads = [W.grad_input(wl, step, 0, scale=orc.state.S)]
        a.step(grads, [10])
        b.step(grads, [10])
        res = orc.step([grad_bits(x) for x in grads], [10], 1.0, **W.HP)
        compare_scalars(b.status(), orc, res, f"resumed step {step}")
    ra, rb = a.pull(), b.pull()
    for k in ra:
        assert np.array_equal(ra[k], rb[k]), k
    for bad in (tl.tl_state(3.0, 0, 0, 1.0, 1.0), tl.tl_state(8.0, 3, 0, 1.0, 1.0),
                tl.tl_state(8.0, 0, -1, 1.0, 1.0), tl.tl_state(0.25, 0, 0, 1.0, 1.0)):
        with pytest.raises(tl.TLError) as ei:
            tl.tl_set_state(b.ctx, bad)
        assert ei.value.status == tl.TL_EINVAL


def test_cuda_graph_capture_replay():
    """The whole update has no host synchronisation, so it can be captured once and
    replayed; replays match eager updates bit for bit."""
    wl = custom([20000, 4099, 8], k=3, steps=4, counts=[3, 1, 2])
    master0 = W.master_init(wl)
    eager = GpuOptimizer(wl, master0)
    graphed = GpuOptimizer(wl, master0, key=30)
    grads = [W.grad_input(wl, 1, i) for i in range(3)]
    pe = [eager.grad_list(i, g) for i, g in enumerate(grads)]
    pg = [graphed.grad_list(i, g) for i, g in enumerate(grads)]
    hp = tl.tl_adamw_hp(**W.HP)
    tl.logical_update(graphed.ctx, pg, [3, 1, 2], 1.0, hp)   # warm-up outside capture
    tl.logical_update(eager.ctx, pe, [3, 1, 2], 1.0, hp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        tl.logical_update(graphed.ctx, pg, [3, 1, 2], 1.0, hp)
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
        tl.logical_update(eager.ctx, pe, [3, 1, 2], 1.0, hp)
    torch.cuda.synchronize()
    re, rg = eager.pull(), graphed.pull()
    for k in re:
        assert np.array_equal(re[k], rg[k]), k
    assert eager.status().t == graphed.status().t == 4


def test_norm_is_deterministic():
    wl = custom([300000, 77, 5000], k=2, steps=1, counts=[1, 1])
    master0 = W.master_init(wl)
    grads = [W.grad_input(wl, 1, i) for i in range(2)]
    norms = []
    for key in (0, 40):
        g = GpuOptimizer(wl, master0, key=key)
        g.step(grads, [1, 1])
        st = g.status()
        norms.append((st.norm, st.sumsq))
    assert norms[0] == norms[1]


class _DeviceScalar:
    """A device address exposed through __cuda_array_interface__ (one fp32)."""

    def __init__(self, addr):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<f4", "data": (addr, False), "version": 2}


def test_scale_pointer_tracks_the_device_scale():
    """tl_scale_ptr lets the loss be scaled on the device; it follows the scaler without a
    host read (here: 8 -> 4 after an overflowing update)."""
    gpu, g = _small_ctx(scaler=True)
    S_dev = torch.as_tensor(_DeviceScalar(tl.tl_scale_ptr(gpu.ctx)), device="cuda")
    loss = torch.tensor([0.75], device="cuda")
    assert float((loss * S_dev).item()) == 6.0
    bad = W.grad_input(gpu.wl, 1, 0, scale=8.0)
    bad.view(torch.int16)[3] = 0x7C00
    gb = gpu.grad_list(1, bad)
    tl.logical_update(gpu.ctx, [gb, gb], [1, 1], 1.0, tl.tl_adamw_hp(**W.HP))
    assert float((loss * S_dev).item()) == 3.0
    assert gpu.status().S == 4.0


def test_loss_seed_follows_the_device_scale():
    """[RST] ch. 13: reverse mode seeded with S * n_i / N (at S = 128, 85.33333333333333 and
    42.666666666666664 for the shares 6/9 and 3/9; here in fp32); after an overflowing update
    the seed halves with S, with no host read of S."""
    wl = custom([64], pdtype="f16", gdtype="f16", k=2, steps=1, counts=[6, 3], scaler=True, init_scale=128.0,
                interval=1000)
    gpu = GpuOptimizer(wl, W.master_init(wl))
    out = torch.zeros(2, dtype=torch.float32, device="cuda")
    tl.tl_loss_seed(gpu.ctx, 6, 9, out.data_ptr())
    tl.tl_loss_seed(gpu.ctx, 3, 9, out.data_ptr() + 4)
    torch.cuda.synchronize()
    assert out[0].item() == np.float32(85.33333333333333) and out[1].item() == np.float32(42.666666666666664)
    bad = W.grad_input(wl, 1, 0, scale=128.0)
    bad.view(torch.int16)[0] = 0x7C00
    gb = gpu.grad_list(0, bad)
    tl.logical_update(gpu.ctx, [gb, gb], [6, 3], 1.0, tl.tl_adamw_hp(**W.HP))
    tl.tl_loss_seed(gpu.ctx, 6, 9, out.data_ptr())
    torch.cuda.synchronize()
    assert out[0].item() == np.float32(85.33333333333333) / 2
    with pytest.raises(tl.TLError) as ei:
        tl.tl_loss_seed(gpu.ctx, 0, 9, out.data_ptr())
    assert ei.value.status == tl.TL_EINVAL


def test_single_tensor_beyond_2_pow_31_full():
    """Maximum-size edge case: one tensor of 2^31 + 77 elements (64-bit chunk offsets)
    next to a 5-element one.  Sampled elements at the start, around element 2^31 and at
    the end against the oracle, one by one; the norm against the fp64 sum of the fp32
    squares computed on the device by torch."""
    import oracle
    n0 = (1 << 31) + 77
    numel = [n0, 5]
    off1 = (n0 + 7) // 8 * 8
    total = off1 + 8
    gen = torch.Generator(device="cuda").manual_seed(31)
    master = torch.randn(total, generator=gen, device="cuda") * 0.02
    param = master.to(torch.bfloat16)
    m = torch.zeros(total, device="cuda")
    v = torch.zeros(total, device="cuda")
    acc = torch.empty(total, device="cuda")
    grads = (torch.randn(total, generator=gen, device="cuda") * 1e-2).to(torch.bfloat16)

    def plist(t):
        es = t.element_size()
        p = tl.PtrList([t.data_ptr(), t.data_ptr() + off1 * es])
        p.keep = t
        return p

    flat_idx = np.concatenate([np.arange(0, 100), np.arange((1 << 31) - 50, (1 << 31) + 50),
                               np.arange(n0 - 100, n0), off1 + np.arange(5)])
    it = torch.from_numpy(flat_idx).cuda()
    w0 = master[it].cpu().numpy()
    gbits = grads[it].cpu().view(torch.int16).numpy().view(np.uint16)
    cfg = tl.make_config(tl.TL_BF16, tl.TL_BF16)
    ctx = tl.tl_create(numel, plist(param), plist(master), plist(m), plist(v), plist(acc), cfg)
    gl = plist(grads)
    tl.logical_update(ctx, [gl], [7], 0.0, tl.tl_adamw_hp(**W.HP))
    st = tl.tl_read_status(ctx)
    assert st.t == 1 and st.skipped == 0 and st.coef == 1.0
    gf = torch.cat([grads[:n0], grads[off1:off1 + 5]]).float()
    ref = float((gf * gf).double().sum())
    del gf
    assert abs(st.sumsq - ref) <= 1e-9 * ref and abs(st.norm - math.sqrt(ref)) <= 1e-6 * math.sqrt(ref)
    lib = oracle.load()
    n = flat_idx.size
    P_ = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    u = np.empty(n, np.float32)
    lib.tlo_accumulate(P_(u), P_(np.ascontiguousarray(gbits)), oracle.DT_BF16, n, lib.tlo_microbatch_weight(7, 7), 1)
    lib.tlo_unscale_check(P_(u), n, 1.0)
    hp = oracle.AdamWHP(**W.HP)
    sc = lib.tlo_adamw_prepare(ctypes.byref(hp), float(np.float32(0.9)), float(np.float32(0.95)))
    w = w0.astype(np.float32).copy()
    mo = np.zeros(n, np.float32)
    vo = np.zeros(n, np.float32)
    po = np.empty(n, np.uint16)
    lib.tlo_adamw_recast(P_(w), P_(mo), P_(vo), P_(po), oracle.DT_BF16, P_(u), n, lib.tlo_clip_coef(st.norm, 0.0),
                         ctypes.byref(sc))
    torch.cuda.synchronize()
    assert_ulps32(master[it].cpu().numpy(), w, 2, "2^31 master")
    assert_ulps32(m[it].cpu().numpy(), mo, 2, "2^31 m")
    assert_ulps32(v[it].cpu().numpy(), vo, 2, "2^31 v")
    assert_ulps16(param[it].cpu().view(torch.int16).numpy().view(np.uint16), po, 1, "2^31 param")


# ---------------------------------------------------------------------------
# the full-size workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("layout,resident", [(True, False), ("packed", False), (False, True), (False, "remat")],
                         ids=["misaligned", "packed", "aligned-resident", "aligned-remat"])
def test_ragged_100k_full(layout, resident):
    """100,000 ragged tensors (~400M parameters) in flat buffers.  Three layouts:
    - independent seeded gaps: most tensors off any 16-byte boundary, so the scalar
      paths run;
    - packed back to back: the same element phase in every list, so the peeled
      vector paths run;
    - every tensor 32-byte aligned, with the resident and the re-materialising
      sequences the benchmark times.
    fp16 with loss scaling and an inf in micro-batch 1 of step 2; every element is
    compared."""
    wl = W.make("ragged_100k")
    _, _, log = run_parity(wl, gaps=layout, compare_every=wl.steps, resident=resident)
    assert [e["skipped"] for e in log] == [0, 1, 0]


@pytest.mark.parametrize("name,resident", [("llama_1b", True), ("llama_1b", False), ("llama_1b_fp8", True)],
                         ids=["bf16-resident", "bf16-per_microbatch", "e4m3b16-resident"])
def test_llama_1b_full_size_sampled(name, resident):
    """The ~1.24B-parameter list at full size, k=8, over the workload's 5 updates, through
    the call sequence the benchmark times (resident: the headline), the per-micro-batch
    sequence, and the resident sequence over 8-bit block-scaled gradients.  Every update:
    the norm against the oracle's sum over every element (the oracle's accumulate and
    unscale run on slices of the list on the host threads, its sum in order), and
    200,000 sampled elements of master, m, v and params advanced one by one through the
    oracle's functions with that update's global clip coefficient, so updates 2-5 read
    non-zero moments back."""
    import oracle
    from harness import oracle_accumulate_par, oracle_dequant_par, oracle_unscale_par
    wl = W.make(name)
    fp8 = wl.grad_dtype == "e4m3b16"
    master0 = W.master_init(wl, "cuda")
    gpu = GpuOptimizer(wl, master0)
    rng = np.random.default_rng(123)
    idx = np.unique(rng.integers(0, wl.P, 200_000))
    idx_t = torch.from_numpy(idx).cuda()
    n = idx.size
    lib = oracle.load()

    def P_(a):
        return a.ctypes.data_as(ctypes.c_void_p)

    # the sampled state, advanced by the oracle's functions
    w = master0[idx_t].cpu().numpy().astype(np.float32).copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    p = np.empty(n, np.uint16)
    state = oracle.State(1.0, 0, 0, 1.0, 1.0)
    scfg = oracle.ScalerCfg(0, 2.0, 0.5, 2000, 1.0, 2.0 ** 127)
    hp = oracle.AdamWHP(**{k: v_ for k, v_ in W.HP.items()})
    acc = np.empty(wl.P, np.float32)
    del master0
    for step in range(1, wl.steps + 1):
        counts = wl.counts(step)
        N = sum(counts)
        grads = [W.grad_input(wl, step, i, device="cuda") for i in range(wl.k)]
        gpu.step(grads, counts, resident=resident)
        st = gpu.status()
        weights = [lib.tlo_microbatch_weight(c, N) for c in counts]
        # the oracle's u over every element, one list at a time (host memory), keeping
        # each list's sampled inputs for the element-wise check below
        samples = []
        for i, g in enumerate(grads):
            if fp8:
                vals = oracle_dequant_par(g[0].cpu().numpy(), g[1].cpu().numpy(), wl.numel)
                dt = oracle.DT_F32
            else:
                vals = np.ascontiguousarray(grad_bits(g))
                dt = oracle.DT_BF16
            oracle_accumulate_par(lib, acc, vals, dt, weights[i], i == 0)
            samples.append((np.ascontiguousarray(vals[idx]), dt))
            del vals
        del grads
        found = oracle_unscale_par(lib, acc, 1.0)
        sumsq = lib.tlo_sumsq(P_(acc), wl.P)
        assert found == 0 and st.found_inf == 0 and st.skipped == 0
        norm = lib.tlo_norm_from_sumsq(sumsq)
        assert abs(st.norm - norm) <= 1e-6 * norm, (step, st.norm, norm)
        coef = lib.tlo_clip_coef(norm, wl.max_norm)
        # sampled elements, one by one, through the oracle's functions in the step's order
        u = np.empty(n, np.float32)
        for i, (vals, dt) in enumerate(samples):
            lib.tlo_accumulate(P_(u), P_(vals), dt, n, weights[i], 1 if i == 0 else 0)
        lib.tlo_unscale_check(P_(u), n, 1.0)
        b1n = state.b1p * float(np.float32(hp.beta1))
        b2n = state.b2p * float(np.float32(hp.beta2))
        sc = lib.tlo_adamw_prepare(ctypes.byref(hp), b1n, b2n)
        lib.tlo_adamw_recast(P_(w), P_(m), P_(v), P_(p), oracle.DT_BF16, P_(u), n, coef, ctypes.byref(sc))
        lib.tlo_scaler_update(ctypes.byref(state), ctypes.byref(scfg), 0, b1n, b2n)
        L = gpu.lists
        what = f"{name} update {step}"
        assert_ulps32(L["master"].flat()[idx_t].cpu().numpy(), w, 2, f"{what} master")
        assert_ulps32(L["m"].flat()[idx_t].cpu().numpy(), m, 2, f"{what} m")
        assert_ulps32(L["v"].flat()[idx_t].cpu().numpy(), v, 2, f"{what} v")
        gp = L["param"].flat()[idx_t].cpu().view(torch.int16).numpy().view(np.uint16)
        assert_ulps16(gp, p, 1, f"{what} param")
        assert st.t == state.t == step and st.b1p == state.b1p and st.b2p == state.b2p
    assert gpu.status().t == 5


@pytest.mark.parametrize("fused", [True, False], ids=["norm_in_pass", "norm_launch"])
def test_failed_launch_abandons_the_update(monkeypatch, fused):
    """Host-side fault injection (no kernel is harmed): the launch of the first AdamW part
    (of two: the small tensor forms a group) reports a failure.  The update in flight is
    abandoned, every update call is refused until tl_set_state restores the scalars, and
    the redone update matches the oracle.  Both with the norm finished by the pass and with
    a separate norm launch (a list of more than 8,192 chunks)."""
    numel = [5000, 300, 17000] if fused else [5000, 300, 17000, 8200 * 16384]
    wl = custom(numel, k=2, steps=1, counts=[3, 4])
    master0 = W.master_init(wl)
    monkeypatch.setenv("TL_SMALL_GROUP_MIN", "1")
    grads = [W.grad_input(wl, 1, i) for i in range(2)]
    # the launches before the AdamW call, counted on a context without the fault
    probe = GpuOptimizer(wl, master0, key=90)
    pp = [probe.grad_list(i, g) for i, g in enumerate(grads)]
    tl.tl_accumulate(probe.ctx, pp[0], 3, 7, 1)
    tl.tl_unscale_check(probe.ctx, pp[1], 4, 7)
    tl.tl_grad_norm(probe.ctx, 1.0)
    before_adamw = tl.tl_launch_count(probe.ctx)
    assert before_adamw == (4 if fused else 5)   # two parts per pass (+ the norm launch)
    del probe, pp
    monkeypatch.setenv("TL_TEST_FAIL_LAUNCH", str(before_adamw + 1))
    gpu = GpuOptimizer(wl, master0)
    monkeypatch.delenv("TL_TEST_FAIL_LAUNCH")
    orc = oracle_for(wl, master0)
    pl = [gpu.grad_list(i, g) for i, g in enumerate(grads)]
    hp = tl.tl_adamw_hp(**W.HP)
    snap = tl.tl_get_state(gpu.ctx)
    tl.tl_accumulate(gpu.ctx, pl[0], 3, 7, 1)
    tl.tl_unscale_check(gpu.ctx, pl[1], 4, 7)
    tl.tl_grad_norm(gpu.ctx, 1.0)
    with pytest.raises(tl.TLError) as ei:
        tl.tl_clip_adamw_step(gpu.ctx, hp)
    assert ei.value.status == tl.TL_ECUDA
    for call in (lambda: tl.tl_scaler_update(gpu.ctx), lambda: tl.tl_accumulate(gpu.ctx, pl[0], 3, 7, 1),
                 lambda: tl.tl_unscale_check_many(gpu.ctx, pl, [3, 4], 7)):
        with pytest.raises(tl.TLError) as ei:
            call()
        assert ei.value.status == tl.TL_ESTATE
    tl.tl_set_state(gpu.ctx, snap)
    tl.logical_update(gpu.ctx, pl, [3, 4], 1.0, hp)
    res = orc.step([grad_bits(g) for g in grads], [3, 4], 1.0, **W.HP)
    compare_scalars(gpu.status(), orc, res, "redone update")
    compare_state(gpu.pull(), orc, wl, "redone update")


def _outside_mask(dl):
    """Positions of a DeviceList buffer that belong to no tensor (gaps, padding, tail)."""
    inside = np.zeros(dl.buf.numel(), dtype=bool)
    for o, n in zip(dl.offs, dl.numel):
        inside[o:o + n] = True
    return torch.from_numpy(~inside).to(dl.buf.device)


@pytest.mark.parametrize("gdtype", ["bf16", "e4m3b16"])
@pytest.mark.parametrize("gaps", [False, True, "packed"], ids=["aligned", "gaps", "packed"])
@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
def test_no_write_outside_tensors(gaps, resident, gdtype):
    """Canary words: every buffer position outside the tensors (gaps between tensors,
    alignment padding, the tail) holds a sentinel before the updates and still holds it
    after them; the gradient buffers are not written at all."""
    wl = custom([1, 7, 9, 127, 1025, 16385, 33, 40000, 8], gdtype=gdtype, k=3, steps=3, counts=[2, 3, 4])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0, gaps=gaps)
    masks = {}
    for name, dl in gpu.lists.items():
        masks[name] = _outside_mask(dl)
        sentinel = 12345.678 if dl.buf.dtype == torch.float32 else -7.5
        dl.buf[masks[name]] = sentinel
    canary = {name: dl.buf[masks[name]].clone() for name, dl in gpu.lists.items()}
    hp = tl.tl_adamw_hp(**W.HP)
    for step in (1, 2, 3):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        pl = [gpu.grad_list(i, g) for i, g in enumerate(grads)]
        before = [gpu.grad_lists[i].buf.clone() for i in range(wl.k)]
        tl.logical_update(gpu.ctx, pl, wl.counts(step), 1.0, hp, resident=resident)
        torch.cuda.synchronize()
        for i in range(wl.k):
            assert torch.equal(gpu.grad_lists[i].buf, before[i]), f"gradient list {i} was written"
    for name, dl in gpu.lists.items():
        assert torch.equal(dl.buf[masks[name]], canary[name]), f"{name}: a write outside the tensors"
