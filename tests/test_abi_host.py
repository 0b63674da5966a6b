"""The C-ABI library on the CPU: it builds, loads, exports every function that
include/tl.h declares, and rejects invalid arguments before touching CUDA
(so these checks run without a GPU).  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tl.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tl_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 16
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (tl_\w+)", out))
    for n in names:
        assert n in exported, n
        getattr(lib, n)
    assert set(tl.EXPORTED) == set(names)


def test_status_strings(lib):
    for code in (tl.TL_OK, tl.TL_EINVAL, tl.TL_ECUDA, tl.TL_ESTATE, tl.TL_ENOMEM):
        assert lib.tl_status_string(code)
    assert lib.tl_last_error(None) == b""


def _create(lib, numel, lists, cfg):
    n = len(numel)
    arr = (ctypes.c_int64 * max(n, 1))(*numel)
    ptrs = [(ctypes.c_void_p * max(n, 1))(*l) for l in lists]
    h = ctypes.c_void_p()
    return lib.tl_create(ctypes.byref(h), n, arr, *ptrs, ctypes.byref(cfg), None)


BASE = 1 << 40  # fake device addresses: validation happens before any CUDA call


def _lists(numel, es_param=2, start=BASE, gap=0):
    out = []
    pos = start
    for es in (es_param, 4, 4, 4, 4):
        lst = []
        for n in numel:
            lst.append(pos)
            pos += n * es + gap
        pos = (pos + 255) // 256 * 256
        out.append(lst)
    return out


def test_create_rejects_invalid_arguments(lib):
    good = tl.make_config(tl.TL_BF16, tl.TL_BF16)
    numel = [10, 20, 30]
    lists = _lists(numel)
    # the valid call gets past validation and only then fails for want of a GPU
    rc_valid = _create(lib, numel, lists, good)
    assert rc_valid in (tl.TL_ECUDA, tl.TL_OK)
    cases = {}
    bad = [l[:] for l in lists]; bad[1][1] = bad[1][0]                       # master tensor passed twice
    cases["duplicate"] = (numel, bad, good)
    bad = [l[:] for l in lists]; bad[2][0] = bad[3][0] + 8                     # m overlaps v
    cases["overlap"] = (numel, bad, good)
    bad = [l[:] for l in lists]; bad[1][2] += 2                                # fp32 not 4-byte aligned
    cases["misaligned"] = (numel, bad, good)
    bad = [l[:] for l in lists]; bad[0][0] += 1                                # bf16 not 2-byte aligned
    cases["misaligned16"] = (numel, bad, good)
    bad = [l[:] for l in lists]; bad[4][1] = 0                                 # NULL acc
    cases["null"] = (numel, bad, good)
    cases["negative_numel"] = ([10, -1, 30], lists, good)
    for name, kw in {"param_dtype": dict(param_dtype=tl.TL_F32), "grad_dtype": dict(grad_dtype=7),
                     "scale_not_pow2": dict(scaler_enabled=True, init_scale=3.0),
                     "growth_not_pow2": dict(scaler_enabled=True, growth=3.0),
                     "backoff_ge_1": dict(scaler_enabled=True, backoff=1.0),
                     "interval_0": dict(scaler_enabled=True, interval=0),
                     "min_gt_max": dict(scaler_enabled=True, min_scale=8.0, max_scale=4.0),
                     "init_below_min": dict(scaler_enabled=True, init_scale=1.0, min_scale=2.0),
                     # a subnormal floor: 1/S would overflow to infinity
                     "min_subnormal": dict(scaler_enabled=True, init_scale=1.0, min_scale=2.0 ** -127)}.items():
        cfg = tl.make_config(**{**dict(param_dtype=tl.TL_BF16, grad_dtype=tl.TL_BF16), **kw})
        cases[name] = (numel, lists, cfg)
    for name, (nm, ls, cfg) in cases.items():
        assert _create(lib, nm, ls, cfg) == tl.TL_EINVAL, name


def test_calls_on_null_context_are_rejected(lib):
    assert lib.tl_accumulate(None, None, 1, 1, 1, None) == tl.TL_EINVAL
    assert lib.tl_unscale_check(None, None, 1, 1, None) == tl.TL_EINVAL
    assert lib.tl_grad_norm(None, 1.0, None) == tl.TL_EINVAL
    assert lib.tl_clip_adamw_step(None, None, None) == tl.TL_EINVAL
    assert lib.tl_scaler_update(None, None) == tl.TL_EINVAL
    assert lib.tl_read_status(None, None, None) == tl.TL_EINVAL
    assert lib.tl_get_state(None, None, None) == tl.TL_EINVAL
    assert lib.tl_set_state(None, None, None) == tl.TL_EINVAL
    assert lib.tl_set_lr_schedule(None, None, 0) == tl.TL_EINVAL
    assert lib.tl_destroy(None) == tl.TL_OK
    assert lib.tl_scale_ptr(None) is None
    assert lib.tl_num_params(None) == 0 and lib.tl_launch_count(None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tl, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(tl, "_lib", None)
    with pytest.raises(ImportError):
        tl.load_library()


def test_product_path_does_not_reach_the_oracle():
    """The package never imports, loads or calls the oracle."""
    pkg = os.path.join(ROOT, "loss_scaled_adamw_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "tlo_" not in text and "libtlo" not in text, f


def test_partition_pieces_match_the_oracle_cut_points(lib):
    """tl_partition (host only): the pieces of every rank, flattened, are exactly the
    oracle's slice [b_r, b_(r+1)), in tensor order, with no empty piece; bad arguments
    are rejected."""
    import numpy as np
    import oracle
    cases = [([37, 4096, 5, 999, 2048, 1, 3000], 2, 16), ([10], 4, 1), ([0, 5, 0, 7], 3, 1),
             ([1] * 50, 7, 1), ([16384] * 8 + [3], 5, 16), ([], 2, 1), ([2 ** 33, 5], 3, 16)]
    for numel, N, align in cases:
        P = sum(numel)
        b = oracle.partition_bounds(P, N, align)
        starts = np.concatenate([[0], np.cumsum(numel)]).astype(np.int64)
        covered = 0
        for r in range(N):
            pieces = tl.tl_partition(numel, N, r, align)
            pos = b[r]
            for t, s, n in pieces:
                assert n > 0 and 0 <= s and s + n <= numel[t]
                assert starts[t] + s == pos            # contiguous, in order
                pos += n
            assert pos == b[r + 1], (numel, N, align, r)
            covered += b[r + 1] - b[r]
        assert covered == P
    arr = (ctypes.c_int64 * 2)(10, 20)
    t, s, n = (ctypes.c_int64 * 2)(), (ctypes.c_int64 * 2)(), (ctypes.c_int64 * 2)()
    cnt = ctypes.c_int64()
    for args in ((2, arr, 0, 0, 1), (2, arr, 2, 2, 1), (2, arr, 2, -1, 1), (2, arr, 2, 0, 0)):
        assert lib.tl_partition(*args, t, s, n, 2, ctypes.byref(cnt)) == tl.TL_EINVAL
    # too small a capacity: the count is still reported
    assert lib.tl_partition(2, arr, 1, 0, 1, t, s, n, 1, ctypes.byref(cnt)) == tl.TL_EINVAL and cnt.value == 2
    assert lib.tl_partition(2, arr, 1, 0, 1, t, s, n, 2, ctypes.byref(cnt)) == tl.TL_OK and cnt.value == 2


def test_sharded_norm_calls_reject_bad_arguments(lib):
    assert lib.tl_local_sumsq(None, None, None, None) == tl.TL_EINVAL
    assert lib.tl_grad_norm_from(None, None, None, 1.0, None) == tl.TL_EINVAL
