"""GPU parity of the re-materialising update (tl_unscale_check_many, then the AdamW
pass recomputing u from the resident lists): against the oracle with the usual
tolerances, and bit for bit against the resident many-list pass that stores u."""
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


@pytest.mark.parametrize("k", [1, 2, 3, 4])
@pytest.mark.parametrize("gaps", [False, True, "packed"], ids=["aligned", "misaligned", "packed"])
def test_remat_parity(k, gaps):
    wl = custom([1, 9, 16385, 5000, 0, 77, 1030, 40000], k=k, steps=2, counts=[3 + (i * 7) % 11 for i in range(k)])
    run_parity(wl, gaps=gaps, resident="remat")


@pytest.mark.parametrize("dtypes", [("f16", "f16"), ("bf16", "f32"), ("f16", "bf16"), ("bf16", "bf16")], ids=str)
def test_remat_dtypes(dtypes):
    wl = custom([4096, 33, 20000, 1025], pdtype=dtypes[0], gdtype=dtypes[1], k=3, steps=2, counts=[1, 2, 3])
    run_parity(wl, gaps=True, resident="remat")


@pytest.mark.parametrize("name", ["bf16_small", "fp16_scaled"])
def test_remat_workloads(name):
    wl = W.make(name)
    run_parity(wl, resident="remat", compare_every=5 if wl.steps > 5 else 1)


@pytest.mark.parametrize("k", [1, 2, 3, 4])
@pytest.mark.parametrize("gdtype", ["bf16", "f32"])
def test_remat_bitwise_equal_to_resident_pass(k, gdtype):
    """Same u (the same operations in the same order), so the same norm and state bit
    for bit; both sides on the same layout."""
    wl = custom([70000, 4099, 123, 8, 16384], gdtype=gdtype, k=k, steps=3, counts=[5, 1, 2, 9][:k])
    master0 = W.master_init(wl)
    a = GpuOptimizer(wl, master0, gaps="packed", key=71)
    b = GpuOptimizer(wl, master0, gaps="packed", key=71)
    for step in (1, 2, 3):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        a.step(grads, wl.counts(step), resident=True)
        b.step(grads, wl.counts(step), resident="remat")
        sa, sb = a.status(), b.status()
        assert (sa.norm, sa.sumsq, sa.coef, sa.t, sa.skipped) == (sb.norm, sb.sumsq, sb.coef, sb.t, sb.skipped)
    ra, rb = a.pull(), b.pull()
    for key in ra:
        assert np.array_equal(ra[key], rb[key]), key


def test_remat_leaves_acc_untouched():
    wl = custom([5000, 300, 17], k=2, steps=1, counts=[4, 5])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0)
    acc = gpu.lists["acc"].buf   # filled with 1e30 when created
    before = acc.clone()
    grads = [W.grad_input(wl, 1, i) for i in range(2)]
    gpu.step(grads, [4, 5], resident="remat")
    torch.cuda.synchronize()
    assert torch.equal(acc, before)


def test_remat_overflow_and_scaler():
    wl = custom([3000, 5000], pdtype="f16", gdtype="f16", k=3, steps=5, counts=[1, 1, 1], scaler=True,
                init_scale=2.0 ** 10, injections={(2, 1): [(10, 0x7C00)], (4, 2): [(4000, 0x7E00)]})
    _, _, log = run_parity(wl, resident="remat")
    assert [e["skipped"] for e in log] == [0, 1, 0, 1, 0]


@pytest.mark.parametrize("ntensors", [257, 600])
def test_remat_long_lists(ntensors):
    """Beyond 256 tensors the k lists travel as cached device pointer tables; the AdamW
    pass finds the same tables again."""
    rng = np.random.default_rng(ntensors)
    wl = custom([int(x) for x in rng.integers(1, 400, ntensors)], k=3, steps=3, counts=[2, 2, 3])
    run_parity(wl, gaps=True, resident="remat")


def test_remat_call_rules():
    wl = custom([5000, 300], k=4, steps=1, counts=[2, 3, 4, 1])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0)
    orc = oracle_for(wl, master0)
    grads = [W.grad_input(wl, 1, i) for i in range(4)]
    pl = [gpu.grad_list(i, g) for i, g in enumerate(grads)]
    hp = tl.tl_adamw_hp(**W.HP)
    extra = gpu.grad_list(4, grads[0])
    for lists, counts, N, code in [
        (pl + [extra], [2, 3, 4, 1, 1], 11, tl.TL_EINVAL),   # more than 4 lists
        (pl, [2, 3, 4, 2], 10, tl.TL_EINVAL),                # counts exceed N
        (pl[:3], [2, 3, 4], 10, tl.TL_EINVAL),               # counts short of N
    ]:
        with pytest.raises(tl.TLError) as ei:
            tl.tl_unscale_check_many(gpu.ctx, lists, counts, N)
        assert ei.value.status == code
    tl.tl_accumulate(gpu.ctx, pl[0], 2, 10, 1)
    with pytest.raises(tl.TLError) as ei:                    # an update is open
        tl.tl_unscale_check_many(gpu.ctx, pl, [2, 3, 4, 1], 10)
    assert ei.value.status == tl.TL_ESTATE
    tl.tl_accumulate(gpu.ctx, pl[0], 2, 10, 1)               # restart: discard the partial update
    with pytest.raises(tl.TLError):
        tl.tl_grad_norm(gpu.ctx, 1.0)                        # the open update has no u yet
    # finish the open update the per-micro-batch way, then a re-materialising one
    tl.tl_accumulate(gpu.ctx, pl[1], 3, 10, 0)
    tl.tl_accumulate(gpu.ctx, pl[2], 4, 10, 0)
    tl.tl_unscale_check(gpu.ctx, pl[3], 1, 10)
    tl.tl_grad_norm(gpu.ctx, 1.0)
    tl.tl_clip_adamw_step(gpu.ctx, hp)
    tl.tl_scaler_update(gpu.ctx)
    orc.step([grad_bits(g) for g in grads], [2, 3, 4, 1], 1.0, **W.HP)
    tl.tl_unscale_check_many(gpu.ctx, pl, [2, 3, 4, 1], 10)
    with pytest.raises(tl.TLError) as ei:                    # u is virtual: nothing may be accumulated onto it
        tl.tl_accumulate(gpu.ctx, pl[0], 2, 10, 0)
    assert ei.value.status == tl.TL_ESTATE
    with pytest.raises(tl.TLError) as ei:
        tl.tl_unscale_check_many(gpu.ctx, pl, [2, 3, 4, 1], 10)
    assert ei.value.status == tl.TL_ESTATE
    tl.tl_grad_norm(gpu.ctx, 1.0)
    tl.tl_clip_adamw_step(gpu.ctx, hp)
    tl.tl_scaler_update(gpu.ctx)
    res = orc.step([grad_bits(g) for g in grads], [2, 3, 4, 1], 1.0, **W.HP)
    compare_scalars(gpu.status(), orc, res, "remat rules")
    compare_state(gpu.pull(), orc, wl, "remat rules")


def test_remat_cuda_graph_replay():
    """The re-materialising update captures like the others; replays match eager
    updates bit for bit."""
    wl = custom([20000, 4099, 8], k=3, steps=4, counts=[3, 1, 2])
    master0 = W.master_init(wl)
    eager = GpuOptimizer(wl, master0)
    graphed = GpuOptimizer(wl, master0, key=30)
    grads = [W.grad_input(wl, 1, i) for i in range(3)]
    pe = [eager.grad_list(i, g) for i, g in enumerate(grads)]
    pg = [graphed.grad_list(i, g) for i, g in enumerate(grads)]
    hp = tl.tl_adamw_hp(**W.HP)
    tl.logical_update(graphed.ctx, pg, [3, 1, 2], 1.0, hp, resident="remat")
    tl.logical_update(eager.ctx, pe, [3, 1, 2], 1.0, hp, resident="remat")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        tl.logical_update(graphed.ctx, pg, [3, 1, 2], 1.0, hp, resident="remat")
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
        tl.logical_update(eager.ctx, pe, [3, 1, 2], 1.0, hp, resident="remat")
    torch.cuda.synchronize()
    re, rg = eager.pull(), graphed.pull()
    for key in re:
        assert np.array_equal(re[key], rg[key]), key
    assert eager.status().t == graphed.status().t == 4
