"""GPU parity of the split forms: on a list of short segments every pass (unscale,
many-list, check, AdamW and its re-materialising form) works four segments per CTA,
64 threads each.  Checked against the oracle for every gradient dtype and sequence,
and bit for bit between the sequences that reach the same u."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W
from harness import GpuOptimizer, run_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def short_list(seed: int, n_big: int = 300, n_small: int = 150):
    """Tensors of 1,025-2,047 elements, each one whole-CTA segment shorter than half of
    the shortest segment length (4,096): the chunk table runs four of them per norm
    partial, which selects the split forms.  Beside them 150 tensors of at most 1,024
    elements (at least 128: the small-tensor groups too)."""
    rng = np.random.default_rng(seed)
    sizes = np.concatenate([rng.integers(1025, 2048, n_big), rng.integers(1, 1025, n_small)])
    rng.shuffle(sizes)
    return [int(x) for x in sizes]


def workload(pdtype, gdtype, k, steps=2, seed=5):
    return W.Workload("split", short_list(seed), pdtype, gdtype, steps=steps, k=k, grad_std=1e-2,
                      scaler_enabled=False, init_scale=1.0, interval=3,
                      fixed_counts=[2 + (i * 5) % 7 for i in range(k)], grads_prescaled=False, injections={})


DTYPES = [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("f16", "bf16"), ("bf16", "e4m3b16")]


@pytest.mark.parametrize("gaps", [False, True], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("resident", [False, True, "remat"], ids=["per_microbatch", "resident", "remat"])
@pytest.mark.parametrize("k", [2, 3])
@pytest.mark.parametrize("dtypes", DTYPES, ids=lambda d: f"{d[0]}-{d[1]}")
def test_split_forms_parity(dtypes, k, resident, gaps):
    """k = 2: the forms of one or two lists (and the rotated form where the lists'
    element phases differ); k = 3: the forms of more lists."""
    run_parity(workload(dtypes[0], dtypes[1], k), gaps=gaps, resident=resident)


@pytest.mark.parametrize("gaps", [False, "packed"], ids=["aligned", "packed"])
@pytest.mark.parametrize("k", [2, 3])
@pytest.mark.parametrize("gdtype", ["bf16", "f32", "e4m3b16"])
def test_split_forms_sequences_agree_bitwise(gdtype, k, gaps):
    """The per-micro-batch, resident and re-materialising sequences reach the same u, and
    where their passes take the same vector plan their split forms sum the same
    elements per lane: the same norm and state bit for bit.  The per-micro-batch and
    resident passes both read the accumulation buffer, so they always plan alike; the
    check pass of the re-materialising sequence does not touch it and plans from the
    gradient lists alone, so it is compared where the buffer and the lists share their
    alignment (not with 8-bit lists in the packed layout, whose codes keep 16-byte gaps
    while the buffer is packed: there its norm may differ from the others in its last
    fp64 bits)."""
    wl = workload("bf16", gdtype, k, steps=3, seed=11)
    master0 = W.master_init(wl)
    paths = (False, True) if (gdtype == "e4m3b16" and gaps == "packed") else (False, True, "remat")
    opts = [GpuOptimizer(wl, master0, gaps=gaps, key=23) for _ in paths]
    for step in (1, 2, 3):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        for opt, resident in zip(opts, paths):
            opt.step(grads, wl.counts(step), resident=resident)
        key = [(s.norm, s.sumsq, s.coef, s.t, s.skipped) for s in (o.status() for o in opts)]
        assert all(x == key[0] for x in key), key
    pulled = [o.pull() for o in opts]
    for name in pulled[0]:
        for other in pulled[1:]:
            assert np.array_equal(pulled[0][name], other[name]), name
