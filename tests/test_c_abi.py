"""include/tl.h from plain C.

CPU: a C99 file that includes the header is compiled with gcc -std=c99 -Wall -Wextra
-Werror -pedantic and linked against the library; it prints the size and the field
offsets of every structure of the interface, which must equal the Python binding's
ctypes mirrors (the binding and a C caller see the same layout).
GPU: a C99 program allocates its own device buffers (cudaMalloc, one per tensor),
drives three logical updates of the 12 x 4,096 bf16 workload through the five calls
and writes the results out; they must match the oracle at the parity tolerances."""
import ctypes
import os
import struct
import subprocess

import numpy as np
import pytest

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CDIR = os.path.join(ROOT, "tests", "c_abi")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
CFLAGS = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I" + os.path.join(ROOT, "include")]


def _link(lib_dir):
    return ["-L" + lib_dir, "-l:libtl_gb300.so", "-Wl,-rpath," + lib_dir]


def test_c99_sees_the_binding_layout(tmp_path):
    _build.build()
    exe = str(tmp_path / "abi_layout")
    subprocess.run(CFLAGS + ["-o", exe, os.path.join(CDIR, "abi_layout.c")] + _link(os.path.dirname(_build.LIB)),
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.strip().splitlines())
    got = {k: int(v) for k, v in got.items()}
    for cls in (tl.tl_config, tl.tl_adamw_hp, tl.tl_state, tl.tl_status, tl.tl_norm_result, tl.tl_plan_info):
        name = cls.__name__
        assert got[name] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[f"{name}.{field}"] == getattr(cls, field).offset, (name, field)
    for c in ("TL_OK", "TL_EINVAL", "TL_ECUDA", "TL_ESTATE", "TL_ENOMEM", "TL_F32", "TL_BF16", "TL_F16", "TL_E4M3B16"):
        assert got[c] == getattr(tl, c), c
    assert got["functions"] == len(tl.EXPORTED)


@pytest.mark.gpu
def test_c_program_runs_updates_through_the_abi(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from loss_scaled_adamw_gb300 import workloads as W
    from harness import compare_state, grad_bits, oracle_for
    _build.build()
    exe = str(tmp_path / "one_update")
    r = subprocess.run(CFLAGS + ["-isystem", os.path.join(CUDA, "include"), "-o", exe,
                                 os.path.join(CDIR, "one_update.c")] + _link(os.path.dirname(_build.LIB)) +
                       ["-L" + os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    wl = W.make("bf16_small")
    master0 = W.master_init(wl)
    orc = oracle_for(wl, master0)
    hp = W.HP
    counts = wl.counts(1)
    blob = [struct.pack("<q", len(wl.numel)), struct.pack(f"<{len(wl.numel)}q", *wl.numel),
            struct.pack("<q", wl.k), struct.pack(f"<{wl.k}q", *counts), struct.pack("<q", wl.steps),
            struct.pack("<6f", hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], wl.max_norm),
            master0.numpy().astype(np.float32).tobytes(),
            W.to_16bit(master0, "bf16").view(torch.int16).numpy().tobytes()]
    results = []
    for step in range(1, wl.steps + 1):
        grads = [W.grad_input(wl, step, i) for i in range(wl.k)]
        blob += [grad_bits(g).tobytes() for g in grads]
        results.append(orc.step([grad_bits(g) for g in grads], counts, wl.max_norm, **hp))
    (tmp_path / "in.bin").write_bytes(b"".join(blob))
    r = subprocess.run([exe, str(tmp_path / "in.bin"), str(tmp_path / "out.bin")], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    raw = (tmp_path / "out.bin").read_bytes()
    P = wl.P
    rec = struct.Struct("<ffdqii")
    for step, res in enumerate(results):
        norm, coef, sumsq, t, skipped, _ = rec.unpack_from(raw, step * rec.size)
        assert skipped == res.skipped == 0 and t == step + 1
        assert abs(norm - res.norm) <= 1e-6 * res.norm and abs(coef - res.coef) <= 2e-6 * res.coef
        assert abs(sumsq - res.sumsq) <= 1e-9 * res.sumsq
    o = wl.steps * rec.size
    f32 = np.frombuffer(raw, dtype=np.float32, count=3 * P, offset=o)
    gpu = {"master": f32[:P], "m": f32[P:2 * P], "v": f32[2 * P:],
           "param": np.frombuffer(raw, dtype=np.uint16, count=P, offset=o + 12 * P)}
    compare_state(gpu, orc, wl, "C program")
