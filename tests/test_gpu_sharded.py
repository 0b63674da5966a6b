"""The sharded optimizer step on one GPU, through the C ABI.

[ZRO] "The scheme": the flattened parameters are split into N slices and each owner
keeps the master weights and moments of its slice alone and updates it; [ZRO]
"Operational sharp edges", "Gradient clipping": each owner sums the squares over its
slice and those scalars are all-reduced before the square root; [MEG] section 6
"Overflow must be global": every owner steps or skips together.  Here the N owners
are N contexts on one GPU over the pieces tl_partition gives them (sub-tensors of one
set of flat buffers); tl_local_sumsq writes each context's squared norm and flag to
device memory, the test combines them on the device (a sum in rank order and a max:
the all-reduces), and tl_grad_norm_from hands the combined values back to every
context.  The result must equal the unsharded GPU update bit for bit (same fp32 norm)
and the oracle's sharded statement within the parity tolerances."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W
from harness import GpuOptimizer, compare_scalars, compare_state, grad_bits, oracle_for

pytestmark = pytest.mark.gpu

NUMEL = [37, 4096, 5, 999, 2048, 1, 3000, 70000, 300]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def _sub(plist, pieces, es):
    """Sub-tensor addresses of the pieces (tensor, start, length) inside a full list."""
    p = tl.PtrList([int(plist.array[t]) + s * es for t, s, _ in pieces])
    p.keep = plist
    return p


@pytest.mark.parametrize("nranks", [2, 3])
@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
def test_sharded_update_matches_unsharded_and_oracle(resident, nranks):
    P = sum(NUMEL)
    inj = {(3, 1): [(P - 5, 0x7C00)]}          # an overflow in the last owner's slice only
    wl = W.Workload("sharded", NUMEL, "f16", "f16", steps=6, k=3, grad_std=3e-2, scaler_enabled=True,
                    init_scale=2.0 ** 10, interval=2, fixed_counts=[3, 1, 2], grads_prescaled=True, injections=inj)
    master0 = W.master_init(wl)
    full = GpuOptimizer(wl, master0)                       # the unsharded update
    sh = GpuOptimizer(wl, master0, key=50)                 # buffers the shards point into
    orc = oracle_for(wl, master0)
    cfg = tl.make_config(tl.TL_F16, tl.TL_F16, True, 2.0 ** 10, interval=2)
    ranks = []
    for r in range(nranks):
        pieces = tl.tl_partition(NUMEL, nranks, r, 16)
        L = sh.lists
        ctx = tl.tl_create([n for _, _, n in pieces], _sub(L["param"].ptrs, pieces, 2),
                           _sub(L["master"].ptrs, pieces, 4), _sub(L["m"].ptrs, pieces, 4),
                           _sub(L["v"].ptrs, pieces, 4), _sub(L["acc"].ptrs, pieces, 4), cfg)
        ranks.append((ctx, pieces))
    sums = torch.zeros(nranks, dtype=torch.float64, device="cuda")
    flags = torch.zeros(nranks, dtype=torch.int32, device="cuda")
    total = torch.zeros(1, dtype=torch.float64, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    hp = tl.tl_adamw_hp(**W.HP)
    counts = [3, 1, 2]
    for step in range(1, wl.steps + 1):
        grads = [W.grad_input(wl, step, i, scale=orc.state.S) for i in range(3)]
        full.step(grads, counts, resident=resident)
        gl = [sh.grad_list(i, g) for i, g in enumerate(grads)]
        for r, (ctx, pieces) in enumerate(ranks):
            mine = [_sub(g, pieces, 2) for g in gl]
            if resident == "remat":
                tl.tl_unscale_check_many(ctx, mine, counts, 6)
            elif resident:
                tl.tl_accumulate_many(ctx, mine, counts, 6, 1)
            else:
                tl.tl_accumulate(ctx, mine[0], 3, 6, 1)
                tl.tl_accumulate(ctx, mine[1], 1, 6, 0)
                tl.tl_unscale_check(ctx, mine[2], 2, 6)
            tl.tl_local_sumsq(ctx, sums[r:].data_ptr(), flags[r:].data_ptr())
        # the all-reduces, on the device: squared norms summed in rank order, flags by max
        acc = sums[0:1].clone()
        for r in range(1, nranks):
            acc = acc + sums[r:r + 1]
        total.copy_(acc)
        flag.copy_(flags.max().reshape(1))
        for ctx, _ in ranks:
            tl.tl_grad_norm_from(ctx, total.data_ptr(), flag.data_ptr(), wl.max_norm)
            tl.tl_clip_adamw_step(ctx, hp)
            tl.tl_scaler_update(ctx)
        res = orc.step([grad_bits(g) for g in grads], counts, wl.max_norm, **W.HP, shards=(nranks, 16))
        ref = full.status()
        torch.cuda.synchronize()
        assert int(flags[-1].item()) == (1 if step == 3 else 0) and not bool(flags[:-1].any())
        for r, (ctx, _) in enumerate(ranks):
            st = tl.tl_read_status(ctx)
            compare_scalars(st, orc, res, f"rank {r} of {nranks} step {step}")
            assert (st.S, st.t, st.skipped, st.count) == (ref.S, ref.t, ref.skipped, ref.count)
            assert st.skipped == (1 if step == 3 else 0)
            if not st.skipped:
                # every rank clips with the global coefficient, equal to the unsharded one
                assert st.norm == ref.norm and st.coef == ref.coef, (st.norm, ref.norm)
                assert abs(st.sumsq - ref.sumsq) <= 1e-12 * ref.sumsq
                assert abs(float(sums[r].item()) - orc.rank_sumsq[r]) <= 1e-9 * orc.rank_sumsq[r]
        a, b = full.pull(), sh.pull()
        for k in a:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), (step, k)
        compare_state(b, orc, wl, f"sharded x{nranks} step {step}")
