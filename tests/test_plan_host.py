"""How the library lays out a tensor list (tl_plan, host only; tl_create takes the same
plan): segment length, small-tensor groups, squared-norm runs, the split forms and the
norm finished in the pass, checked from the sizes by counting, on the CPU."""
import math

import pytest

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W

CHUNK, MIN_SEG, SEG_PER_SM, SMALL, GROUP, RUN, GROUP_MIN, FUSE_MAX = 16384, 4096, 24, 1024, 8, 4, 128, 8192


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def expected(numel, sm=152):
    """The rules restated: the segment length is the longest power of two from 16,384
    down to 4,096 that gives the whole-CTA part at least 24 segments per SM; tensors of
    at most 1,024 elements go 8 to a group when there are at least 128 of them; runs of
    4 chunks where the whole-CTA segments average under half a segment; tables of at
    most 8,192 chunks finish the norm in the pass."""
    sizes = [n for n in numel if n > 0]
    small = [n for n in sizes if n <= SMALL]
    grouping = len(small) >= GROUP_MIN
    whole = sum(sizes) - (sum(small) if grouping else 0)
    seg = CHUNK
    while seg > MIN_SEG and whole // seg < SEG_PER_SM * sm:
        seg //= 2
    big = [n for n in sizes if not (grouping and n <= SMALL)]
    nbig = sum(math.ceil(n / seg) for n in big)
    ngroups = math.ceil(len(small) / GROUP) if grouping else 0
    run_big = RUN if nbig > 0 and sum(big) < nbig * (seg // 2) else 1
    nchunks = nbig + ngroups
    return {"nchunks": nchunks, "nbig": nbig, "ngroups": ngroups, "seg": seg,
            "nsmall": len(small) if grouping else 0, "run_big": run_big, "run_small": RUN,
            "split_forms": int(run_big > 1), "fused_norm": int(0 < nchunks <= FUSE_MAX)}


@pytest.mark.parametrize("name", ["llama_1b", "llama_10m", "ragged_100k", "bf16_small", "fp16_scaled",
                                  "fp8_small", "stream_64m", "ragged_25k"])
def test_plan_of_the_workloads(name):
    numel = W.make(name).numel
    assert tl.tl_plan(numel) == expected(numel)


def test_plan_figures_the_measurements_rely_on():
    """The layouts the benchmark's workloads are described with: the 1.24B list in full
    segments, one partial per chunk and a separate reduce; the 10M list in 4,096-element
    segments with the norm finished in the pass; the ragged list's 50,094 segments in
    the split forms beside 7,910 groups of its 63,279 small tensors."""
    p = tl.tl_plan(W.make("llama_1b").numel)
    assert (p["seg"], p["ngroups"], p["run_big"], p["split_forms"], p["fused_norm"]) == (16384, 0, 1, 0, 0)
    p = tl.tl_plan(W.make("llama_10m").numel)
    assert (p["seg"], p["nchunks"], p["fused_norm"], p["split_forms"]) == (4096, 2561, 1, 0)
    p = tl.tl_plan(W.make("ragged_100k").numel)
    assert (p["nbig"], p["ngroups"], p["nsmall"], p["run_big"], p["split_forms"], p["fused_norm"]) == \
        (50094, 7910, 63279, 4, 1, 0)


def test_split_form_test_list_selects_the_split_forms():
    """The list of the split-form GPU tests (single-segment tensors of 1,025-2,047
    elements beside 150 small ones) takes the split forms and the groups."""
    import numpy as np
    rng = np.random.default_rng(5)
    sizes = np.concatenate([rng.integers(1025, 2048, 300), rng.integers(1, 1025, 150)])
    p = tl.tl_plan([int(x) for x in sizes])
    assert p["split_forms"] == 1 and p["run_big"] == 4 and p["ngroups"] == math.ceil(150 / 8)


def test_segment_length_follows_the_sm_count():
    numel = [10_000_000]
    assert tl.tl_plan(numel, 152)["seg"] == 4096      # 2,441 segments of 4,096 < 24 x 152 still: floor
    assert tl.tl_plan(numel, 8)["seg"] == 16384       # 610 segments >= 24 x 8
    assert tl.tl_plan(numel, 20)["seg"] == 16384
    assert tl.tl_plan(numel, 26)["seg"] == 8192       # 610 < 624: halve once
    for sm in (1, 7, 26, 100, 152, 1000):
        assert tl.tl_plan(numel, sm) == expected(numel, sm)


def test_grouping_threshold_and_override(monkeypatch):
    few = [100] * 127 + [50_000]
    many = [100] * 128 + [50_000]
    # a list this small takes the shortest segment: 13 segments of the large tensor
    assert tl.tl_plan(few)["ngroups"] == 0 and tl.tl_plan(few)["nbig"] == 127 + math.ceil(50_000 / MIN_SEG)
    assert tl.tl_plan(many)["ngroups"] == 16 and tl.tl_plan(many)["nsmall"] == 128
    monkeypatch.setenv("TL_SMALL_GROUP_MIN", "1")
    assert tl.tl_plan([100, 50_000])["ngroups"] == 1


def test_fused_norm_threshold_and_edges():
    at = [CHUNK] * FUSE_MAX
    assert tl.tl_plan(at)["fused_norm"] == 1
    assert tl.tl_plan(at + [CHUNK])["fused_norm"] == 0
    assert tl.tl_plan([]) == expected([])
    assert tl.tl_plan([0, 0]) == expected([0, 0]) and tl.tl_plan([0, 0])["nchunks"] == 0
    assert tl.tl_plan([1]) == expected([1])


def test_plan_rejects_bad_arguments():
    import ctypes
    lib = tl.load_library()
    out = tl.tl_plan_info()
    arr = (ctypes.c_int64 * 2)(5, -1)
    assert lib.tl_plan(2, arr, 152, ctypes.byref(out)) == tl.TL_EINVAL        # negative size
    arr = (ctypes.c_int64 * 2)(5, 6)
    assert lib.tl_plan(2, arr, 0, ctypes.byref(out)) == tl.TL_EINVAL          # no SMs
    assert lib.tl_plan(-1, arr, 152, ctypes.byref(out)) == tl.TL_EINVAL
    assert lib.tl_plan(2, None, 152, ctypes.byref(out)) == tl.TL_EINVAL
    assert lib.tl_plan(2, arr, 152, None) == tl.TL_EINVAL
    assert lib.tl_plan(2, arr, 152, ctypes.byref(out)) == tl.TL_OK and out.nchunks == 2
