"""GPU parity of the many-list pass (tl_accumulate_many): all k resident micro-batch
gradient lists read in one pass.  Against the oracle with the same tolerances as the
per-micro-batch path, and bit for bit against that path on the same inputs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W
from harness import GpuOptimizer, compare_scalars, compare_state, grad_bits, oracle_for, run_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def custom(numel, pdtype="bf16", gdtype="bf16", k=2, steps=2, counts=None, scaler=False, init_scale=1.0,
           injections=None):
    return W.Workload("custom", list(numel), pdtype, gdtype, steps=steps, k=k, grad_std=1e-2, scaler_enabled=scaler,
                      init_scale=init_scale, interval=3, fixed_counts=counts, grads_prescaled=scaler,
                      injections=injections or {})


@pytest.mark.parametrize("name", ["bf16_small", "fp16_scaled", "llama_10m"])
def test_workloads_resident(name):
    wl = W.make(name)
    run_parity(wl, resident=True, compare_every=5 if wl.steps > 5 else 1)


@pytest.mark.parametrize("k", [1, 2, 3, 8, 9, 10, 11, 17])
@pytest.mark.parametrize("gaps", [False, True, "packed"], ids=["aligned", "misaligned", "packed"])
def test_micro_batch_counts_resident(k, gaps):
    wl = custom([1, 9, 16385, 5000, 0, 77], k=k, steps=2, counts=[3 + (i * 7) % 11 for i in range(k)])
    run_parity(wl, gaps=gaps, resident=True)


@pytest.mark.parametrize("k", [2, 4])
@pytest.mark.parametrize("dtypes", [("f16", "f16"), ("bf16", "f32"), ("f16", "bf16")], ids=str)
def test_dtypes_resident(dtypes, k):
    wl = custom([4096, 33, 20000], pdtype=dtypes[0], gdtype=dtypes[1], k=k, steps=2, counts=[1, 2, 3, 4][:k])
    run_parity(wl, gaps=True, resident=True)


@pytest.mark.parametrize("split", [(2, 2), (1, 3), (3, 1), (2, 1, 1), (1, 1, 1, 1)], ids=str)
@pytest.mark.parametrize("gdtype", ["bf16", "f16", "f32"])
def test_split_resident_calls(split, gdtype):
    """One update fed by several tl_accumulate_many calls of one to three lists (the
    launches of at most two lists take a kernel form of their own, with and without
    a partial sum already in the buffer, and with and without the unscale); bit for
    bit equal to the per-micro-batch path, and within tolerance of the oracle."""
    pdtype = "f16" if gdtype == "f16" else "bf16"
    wl = custom([70000, 4099, 123, 8, 16384], pdtype=pdtype, gdtype=gdtype, k=4, steps=2, counts=[5, 1, 2, 9])
    master0 = W.master_init(wl)
    # the same layout for both: which elements a thread sums (so the last bits of
    # the squared norm) depends on the alignment of the lists
    a = GpuOptimizer(wl, master0, gaps="packed", key=61)
    b = GpuOptimizer(wl, master0, gaps="packed", key=61)
    orc = oracle_for(wl, master0)
    hp = tl.tl_adamw_hp(**W.HP)
    for step in (1, 2):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        counts = wl.counts(step)
        a.step(grads, counts, resident=False)
        pl = [b.grad_list(i, g) for i, g in enumerate(grads)]
        j = 0
        for n in split:
            tl.tl_accumulate_many(b.ctx, pl[j:j + n], counts[j:j + n], sum(counts), int(j + n == wl.k))
            j += n
        tl.tl_grad_norm(b.ctx, wl.max_norm)
        tl.tl_clip_adamw_step(b.ctx, hp)
        tl.tl_scaler_update(b.ctx)
        res = orc.step([grad_bits(g) for g in grads], counts, wl.max_norm, **W.HP)
        sa, sb = a.status(), b.status()
        assert (sa.norm, sa.sumsq, sa.coef, sa.t) == (sb.norm, sb.sumsq, sb.coef, sb.t)
        compare_scalars(sb, orc, res, f"split {split} step {step}")
    ra, rb = a.pull(), b.pull()
    for key in ra:
        assert np.array_equal(ra[key], rb[key]), key
    compare_state(rb, orc, wl, f"split {split}")


@pytest.mark.parametrize("ntensors", [256, 257, 600])
def test_long_lists_resident(ntensors):
    """Past 256 tensors the k lists use cached device pointer tables."""
    rng = np.random.default_rng(ntensors)
    wl = custom([int(x) for x in rng.integers(1, 400, ntensors)], k=5, steps=3, counts=[2, 2, 3, 1, 5])
    run_parity(wl, gaps=True, resident=True)


def test_overflow_and_scaler_resident():
    wl = custom([3000, 5000], pdtype="f16", gdtype="f16", k=3, steps=5, counts=[1, 1, 1], scaler=True,
                init_scale=2.0 ** 10, injections={(2, 1): [(10, 0x7C00)], (4, 2): [(4000, 0x7E00)]})
    _, _, log = run_parity(wl, resident=True)
    assert [e["skipped"] for e in log] == [0, 1, 0, 1, 0]


def test_bitwise_equal_to_per_micro_batch_path():
    wl = custom([70000, 4099, 123, 8], k=6, steps=3, counts=[5, 1, 2, 9, 3, 3])
    master0 = W.master_init(wl)
    a = GpuOptimizer(wl, master0, gaps=True)
    b = GpuOptimizer(wl, master0, gaps=True, key=60)
    for step in (1, 2, 3):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        a.step(grads, wl.counts(step), resident=False)
        b.step(grads, wl.counts(step), resident=True)
        sa, sb = a.status(), b.status()
        assert (sa.norm, sa.sumsq, sa.coef, sa.t) == (sb.norm, sb.sumsq, sb.coef, sb.t)
    ra, rb = a.pull(), b.pull()
    for k in ra:
        assert np.array_equal(ra[k], rb[k]), k


def test_mixed_with_single_accumulate_and_errors():
    """An update may start with tl_accumulate and finish with tl_accumulate_many; counts that
    do not add up are rejected before any launch."""
    wl = custom([5000, 300], k=4, steps=1, counts=[2, 3, 4, 1])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0)
    orc = oracle_for(wl, master0)
    grads = [W.grad_input(wl, 1, i) for i in range(4)]
    pl = [gpu.grad_list(i, g) for i, g in enumerate(grads)]
    N = 10
    with pytest.raises(tl.TLError) as ei:
        tl.tl_accumulate_many(gpu.ctx, pl, [2, 3, 4, 2], N, 1)   # 11 != 10
    assert ei.value.status == tl.TL_EINVAL
    with pytest.raises(tl.TLError) as ei:
        tl.tl_accumulate_many(gpu.ctx, pl[:2], [2, 3], N, 1)     # last, but only 5 of 10
    assert ei.value.status == tl.TL_EINVAL
    tl.tl_accumulate(gpu.ctx, pl[0], 2, N, 1)
    tl.tl_accumulate_many(gpu.ctx, pl[1:3], [3, 4], N, 0)
    tl.tl_accumulate_many(gpu.ctx, pl[3:], [1], N, 1)
    with pytest.raises(tl.TLError) as ei:
        tl.tl_accumulate_many(gpu.ctx, pl[3:], [1], N, 1)
    assert ei.value.status == tl.TL_ESTATE
    tl.tl_grad_norm(gpu.ctx, 1.0)
    tl.tl_clip_adamw_step(gpu.ctx, tl.tl_adamw_hp(**W.HP))
    tl.tl_scaler_update(gpu.ctx)
    res = orc.step([grad_bits(g) for g in grads], [2, 3, 4, 1], 1.0, **W.HP)
    compare_scalars(gpu.status(), orc, res, "mixed")
    compare_state(gpu.pull(), orc, wl, "mixed")
