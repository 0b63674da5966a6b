"""GPU parity of the learning-rate schedule read on the device (tl_set_lr_schedule).

The rate of the update that would commit optimizer step t+1 is the schedule's entry
for that step, t counting committed steps only. An update skipped on overflow
therefore leaves the next rate for the next attempt: in the Rust chapter's
"Discard a failed partial logical update", the optimizer step stays and the
scheduled step remains available. Past the end of the table the last entry holds.
Every test compares with the oracle, which applies the same rule."""
import ctypes

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
           interval=3, injections=None):
    return W.Workload("custom", list(numel), pdtype, gdtype, steps=steps, k=k, grad_std=1e-2, scaler_enabled=scaler,
                      init_scale=init_scale, interval=interval, fixed_counts=counts, grads_prescaled=scaler,
                      injections=injections or {})


# linear warm-up, then decay; distinct rates, shorter than the runs below
SCHEDULE = np.array([2e-4, 4e-4, 6e-4, 8e-4, 1e-3, 7e-4, 4e-4], np.float32)


@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
def test_schedule_with_skipped_updates(resident):
    """fp16 with dynamic scaling and two overflowing updates among ten: the rates follow
    the committed steps, and the last entry holds past the end of the table."""
    wl = custom([5000, 33, 16385, 700], pdtype="f16", gdtype="f16", k=2, steps=10, counts=[3, 5], scaler=True,
                init_scale=2.0 ** 10, injections={(3, 1): [(7, 0x7C00)], (6, 0): [(20000, 0x7E00)]})
    _, orc, log = run_parity(wl, gaps=True, resident=resident, lr_schedule=SCHEDULE)
    assert [e["skipped"] for e in log] == [0, 0, 1, 0, 0, 1, 0, 0, 0, 0]
    assert orc.state.t == 8 > SCHEDULE.size


def test_schedule_in_cuda_graph():
    """Captured once, the update follows the schedule on every replay (the rate is chosen
    on the device from the step count), and a table entry rewritten between replays, in
    stream order, is the one the next replay uses."""
    wl = custom([20000, 4099, 8], k=3, steps=1, counts=[3, 1, 2])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0)
    orc = oracle_for(wl, master0)
    grads = [W.grad_input(wl, 1, i) for i in range(3)]
    ptrs = [gpu.grad_list(i, g) for i, g in enumerate(grads)]
    bits = [grad_bits(g) for g in grads]
    table = torch.from_numpy(SCHEDULE.copy()).cuda()
    tl.tl_set_lr_schedule(gpu.ctx, table)
    host_table = SCHEDULE.copy()
    hp = tl.tl_adamw_hp(**W.HP)
    tl.logical_update(gpu.ctx, ptrs, [3, 1, 2], wl.max_norm, hp)   # warm-up outside capture
    orc.step(bits, [3, 1, 2], wl.max_norm, **W.HP, lr_schedule=host_table)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        tl.logical_update(gpu.ctx, ptrs, [3, 1, 2], wl.max_norm, hp)
    torch.cuda.synchronize()
    for r in range(9):
        if r == 3:
            table[4].fill_(3e-3)          # the rate of step 5, before the replay that commits it
            host_table[4] = np.float32(3e-3)
        graph.replay()
        res = orc.step(bits, [3, 1, 2], wl.max_norm, **W.HP, lr_schedule=host_table)
        compare_scalars(gpu.status(), orc, res, f"replay {r}")
    compare_state(gpu.pull(), orc, wl, "after the replays")
    assert orc.state.t == 10


def test_schedule_removed_and_restored_step():
    """Removing the schedule brings hp.lr back; a state restored with another step count
    reads the schedule from that step on."""
    wl = custom([9000, 130, 1], k=2, steps=1, counts=[2, 7])
    master0 = W.master_init(wl)
    gpu = GpuOptimizer(wl, master0)
    orc = oracle_for(wl, master0)
    table = torch.from_numpy(SCHEDULE.copy()).cuda()
    tl.tl_set_lr_schedule(gpu.ctx, table)
    plan = ["sched", "sched", "none", "none", "restore", "sched", "sched"]
    for step, what in enumerate(plan, start=1):
        if what == "none" and gpu.ctx.lr_table is not None:
            tl.tl_set_lr_schedule(gpu.ctx, None)
        if what == "restore":
            # resume from the optimizer scalars of a checkpoint taken after step 1
            st = tl.tl_get_state(gpu.ctx)
            st.t = 1
            st.b1p = float(np.float32(W.HP["beta1"]))
            st.b2p = float(np.float32(W.HP["beta2"]))
            tl.tl_set_state(gpu.ctx, st)
            orc.state.t, orc.state.b1p, orc.state.b2p = st.t, st.b1p, st.b2p
            tl.tl_set_lr_schedule(gpu.ctx, table)
        grads = [W.grad_input(wl, step, i) for i in range(2)]
        gpu.step(grads, [2, 7])
        kw = {} if what == "none" else {"lr_schedule": SCHEDULE}
        res = orc.step([grad_bits(g) for g in grads], [2, 7], wl.max_norm, **W.HP, **kw)
        compare_scalars(gpu.status(), orc, res, f"step {step} ({what})")
        compare_state(gpu.pull(), orc, wl, f"step {step} ({what})")
    assert orc.state.t == 4


def test_schedule_rejects_bad_arguments():
    wl = custom([100], k=1, steps=1, counts=[1])
    gpu = GpuOptimizer(wl, W.master_init(wl))
    lib = tl.load_library()
    table = torch.zeros(4, dtype=torch.float32, device="cuda")
    assert lib.tl_set_lr_schedule(gpu.ctx.handle, None, -1) == tl.TL_EINVAL
    assert lib.tl_set_lr_schedule(gpu.ctx.handle, None, 3) == tl.TL_EINVAL
    assert lib.tl_set_lr_schedule(gpu.ctx.handle, ctypes.c_void_p(table.data_ptr() + 2), 2) == tl.TL_EINVAL
    with pytest.raises(ValueError):
        tl.tl_set_lr_schedule(gpu.ctx, table.double())
    # the rejected calls left no schedule behind: hp.lr applies
    orc = oracle_for(wl, W.master_init(wl))
    grads = [W.grad_input(wl, 1, 0)]
    gpu.step(grads, [1])
    res = orc.step([grad_bits(grads[0])], [1], wl.max_norm, **W.HP)
    compare_scalars(gpu.status(), orc, res, "no schedule")
    compare_state(gpu.pull(), orc, wl, "no schedule")
