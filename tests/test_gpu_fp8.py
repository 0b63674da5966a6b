"""GPU parity of 8-bit gradients with fine-grained scaling ("Training at Scale",
section 41.5: E4M3 codes with one fp32 scale per block of 16, dequantized before
accumulation) through every path of the update, against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W
from harness import E4M3DeviceList, GpuOptimizer, compare_scalars, compare_state, grad_bits, oracle_for, run_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def fp8(numel, k=2, steps=2, counts=None, pdtype="bf16", injections=None, scaler=False, init_scale=1.0):
    return W.Workload("fp8", list(numel), pdtype, "e4m3b16", steps=steps, k=k, grad_std=1e-2,
                      scaler_enabled=scaler, init_scale=init_scale, interval=3, fixed_counts=counts,
                      grads_prescaled=scaler, injections=injections or {})


@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
@pytest.mark.parametrize("gaps", [False, True], ids=["aligned", "gaps"])
def test_fp8_small(resident, gaps):
    wl = W.make("fp8_small")
    _, _, log = run_parity(wl, gaps=gaps, resident=resident)
    assert [e["skipped"] for e in log] == [0, 0, 1, 0]


@pytest.mark.parametrize("k", [1, 2, 3, 5, 9])
def test_fp8_edge_lists(k):
    """Tensors of 1, 15, 16, 17, 31, 33 elements (partial and single blocks), one
    segment boundary (16,384 / 16,385) and a long tensor, every path that takes k lists."""
    wl = fp8([1, 15, 16, 17, 31, 33, 16384, 16385, 40000], k=k, steps=2,
             counts=[2 + (i * 5) % 7 for i in range(k)])
    run_parity(wl, resident=False)
    run_parity(wl, resident=True)
    if k <= 4:
        run_parity(wl, resident="remat")


def test_fp8_fp16_params_and_scaler():
    wl = fp8([5000, 300, 4096], k=2, steps=5, counts=[3, 4], pdtype="f16", scaler=True, init_scale=2.0 ** 8,
             injections={(2, 1): [(10, 0x7F)], (4, 0): [(9000, 0xFF)]})
    _, _, log = run_parity(wl, resident=True)
    assert [e["skipped"] for e in log] == [0, 1, 0, 1, 0]


@pytest.mark.parametrize("ntensors", [300, 700])
def test_fp8_long_lists(ntensors):
    """Beyond the by-value limits the lists travel as cached device pointer tables."""
    rng = np.random.default_rng(ntensors)
    wl = fp8([int(x) for x in rng.integers(1, 600, ntensors)], k=3, steps=2, counts=[2, 2, 3])
    run_parity(wl, gaps=True, resident=True)
    run_parity(wl, gaps=True, resident=False)


def test_fp8_resident_equals_per_microbatch_bitwise():
    wl = fp8([70000, 4099, 123, 8, 16384], k=6, steps=2, counts=[5, 1, 2, 9, 3, 3])
    master0 = W.master_init(wl)
    a = GpuOptimizer(wl, master0)
    b = GpuOptimizer(wl, master0)
    for step in (1, 2):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        a.step(grads, wl.counts(step), resident=False)
        b.step(grads, wl.counts(step), resident=True)
        sa, sb = a.status(), b.status()
        assert (sa.norm, sa.sumsq, sa.coef) == (sb.norm, sb.sumsq, sb.coef)
    ra, rb = a.pull(), b.pull()
    for key in ra:
        assert np.array_equal(ra[key], rb[key]), key


def test_fp8_pointer_rules():
    """8-bit gradient tensors must start on 16-byte boundaries and must not overlap a state
    tensor (codes, padding and scales all count); violations are rejected before launch."""
    wl = fp8([100, 40], k=1, steps=1, counts=[4])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0)
    g = W.grad_input(wl, 1, 0)
    good = gpu.grad_list(0, g)
    base = [int(x) for x in good.array]
    bad = tl.PtrList([base[0] + 8, base[1]])
    bad.keep = good
    with pytest.raises(tl.TLError) as ei:
        tl.tl_unscale_check(gpu.ctx, bad, 4, 4)
    assert ei.value.status == tl.TL_EINVAL
    acc_end = int(gpu.lists["acc"].ptrs.array[0])        # a "gradient" ending inside the acc list
    over = tl.PtrList([acc_end - 112, base[1]])
    over.keep = good
    with pytest.raises(tl.TLError) as ei:
        tl.tl_unscale_check(gpu.ctx, over, 4, 4)
    assert ei.value.status == tl.TL_EINVAL
    tl.tl_unscale_check(gpu.ctx, good, 4, 4)
    tl.tl_grad_norm(gpu.ctx, 1.0)
    tl.tl_clip_adamw_step(gpu.ctx, tl.tl_adamw_hp(**W.HP))
    tl.tl_scaler_update(gpu.ctx)
    orc = oracle_for(wl, master0)
    res = orc.step([grad_bits(g)], [4], wl.max_norm, **W.HP)
    compare_scalars(gpu.status(), orc, res, "fp8 rules")
    compare_state(gpu.pull(), orc, wl, "fp8 rules")
