"""The oracle: a plain CPU statement of the loss-scaled AdamW optimizer step.

TEST INFRASTRUCTURE ONLY.  The arithmetic lives in ``tlo.c`` (plain C, every
operation an explicit IEEE binary32/binary64 operation, compiled with
``-ffp-contract=off``); this module compiles it with gcc and exposes it through
ctypes over numpy arrays.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package.  It imports
nothing from the GPU library and the GPU library imports nothing from it.

Parity status of each function (what pins it is listed in tests/test_oracle_pins.py):
all functions are pinned; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tlo.c")
_LIB_PATH = os.path.join(_HERE, "libtlo.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

DT_F32, DT_BF16, DT_F16, DT_E4M3B16 = 0, 1, 2, 3
_DT_BY_NAME = {"f32": DT_F32, "bf16": DT_BF16, "f16": DT_F16, "e4m3b16": DT_E4M3B16}


class E4M3List(ctypes.Structure):
    """One micro-batch of 8-bit gradients: E4M3 codes of every tensor back to back and
    each tensor's ceil(numel/16) fp32 block scales back to back."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("numel", ctypes.c_void_p),
                ("ntensors", ctypes.c_int64)]

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB_PATH, extra_cflags=()) -> str:
    """Compile an oracle C source into a shared library with gcc."""
    cmd = ["gcc", *CFLAGS, *extra_cflags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build() -> str:
    """Build libtlo.so next to this file if it is missing or older than tlo.c."""
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        compile_library(out=tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class AdamWHP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class AdamWScalars(ctypes.Structure):
    _fields_ = [("step_size", ctypes.c_float), ("bc2_sqrt", ctypes.c_float), ("lr_wd", ctypes.c_float),
                ("beta1", ctypes.c_float), ("one_minus_beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("one_minus_beta2", ctypes.c_float), ("eps", ctypes.c_float)]


class ScalerCfg(ctypes.Structure):
    _fields_ = [("enabled", ctypes.c_int), ("growth", ctypes.c_float), ("backoff", ctypes.c_float),
                ("interval", ctypes.c_int32), ("min_scale", ctypes.c_float), ("max_scale", ctypes.c_float)]


class State(ctypes.Structure):
    _fields_ = [("S", ctypes.c_float), ("count", ctypes.c_int32), ("t", ctypes.c_int64),
                ("b1p", ctypes.c_double), ("b2p", ctypes.c_double)]


class Result(ctypes.Structure):
    _fields_ = [("skipped", ctypes.c_int), ("found_inf", ctypes.c_int), ("norm", ctypes.c_float),
                ("coef", ctypes.c_float), ("sumsq", ctypes.c_double)]


def _bind(lib):
    vp, i64, f32, f64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_int
    u16 = ctypes.c_uint16
    sig = {
        "tlo_bf16_to_f32": (f32, [u16]),
        "tlo_f16_to_f32": (f32, [u16]),
        "tlo_f32_to_bf16": (u16, [f32]),
        "tlo_f32_to_f16": (u16, [f32]),
        "tlo_decode16": (None, [vp, vp, i64, i32]),
        "tlo_e4m3_to_f32": (f32, [ctypes.c_uint8]),
        "tlo_dequant_e4m3b16": (None, [ctypes.POINTER(E4M3List), vp]),
        "tlo_recast": (None, [vp, vp, i64, i32]),
        "tlo_microbatch_weight": (f32, [i64, i64]),
        "tlo_accumulate": (None, [vp, vp, i32, i64, f32, i32]),
        "tlo_unscale_check": (i32, [vp, i64, f32]),
        "tlo_sumsq": (f64, [vp, i64]),
        "tlo_norm_from_sumsq": (f32, [f64]),
        "tlo_clip_coef": (f32, [f32, f32]),
        "tlo_scheduled_lr": (f32, [vp, i64, i64]),
        "tlo_adamw_prepare": (AdamWScalars, [ctypes.POINTER(AdamWHP), f64, f64]),
        "tlo_adamw_recast": (None, [vp, vp, vp, vp, i32, vp, i64, f32, ctypes.POINTER(AdamWScalars)]),
        "tlo_scaler_update": (None, [ctypes.POINTER(State), ctypes.POINTER(ScalerCfg), i32, f64, f64]),
        "tlo_step": (i32, [vp, vp, vp, vp, i32, vp, i64, ctypes.POINTER(vp), i32, ctypes.POINTER(i64), i32,
                           f32, ctypes.POINTER(AdamWHP), ctypes.POINTER(ScalerCfg), ctypes.POINTER(State),
                           ctypes.POINTER(Result)]),
        "tlo_partition_bounds": (None, [i64, i32, i64, vp]),
        "tlo_step_sharded": (i32, [vp, vp, vp, vp, i32, vp, i64, ctypes.POINTER(vp), i32, ctypes.POINTER(i64), i32,
                                   f32, ctypes.POINTER(AdamWHP), ctypes.POINTER(ScalerCfg), ctypes.POINTER(State),
                                   ctypes.POINTER(Result), i32, i64, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  With ``path`` given, load
    that library instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def dtype_code(name: str) -> int:
    return _DT_BY_NAME[name]


class Oracle:
    """The oracle's optimizer: fp32 master/m/v, a 16-bit model copy, the fp32
    accumulation buffer and the scaler state, all over flat numpy arrays (the
    flattened tensor list, in tensor order)."""

    def __init__(self, master: np.ndarray, param_bits: np.ndarray, param_dtype: str = "bf16",
                 grad_dtype: str = "bf16", scaler_enabled: bool = False, init_scale: float = 1.0,
                 growth: float = 2.0, backoff: float = 0.5, interval: int = 2000,
                 min_scale: float = 1.0, max_scale: float = 2.0 ** 127, lib=None, numel=None):
        self.lib = lib if lib is not None else load()
        # the tensor sizes, needed to place the block scales of 8-bit gradients
        self.numel = None if numel is None else np.ascontiguousarray(numel, dtype=np.int64)
        self.w = np.ascontiguousarray(master, dtype=np.float32).copy()
        self.m = np.zeros_like(self.w)
        self.v = np.zeros_like(self.w)
        self.p = np.ascontiguousarray(param_bits, dtype=np.uint16).copy()
        self.acc = np.zeros_like(self.w)
        self.pdtype = _DT_BY_NAME[param_dtype]
        self.gdtype = _DT_BY_NAME[grad_dtype]
        self.cfg = ScalerCfg(1 if scaler_enabled else 0, growth, backoff, interval, min_scale, max_scale)
        self.state = State(init_scale if scaler_enabled else 1.0, 0, 0, 1.0, 1.0)
        self.last = Result()

    @property
    def P(self) -> int:
        return int(self.w.size)

    def step(self, grads, counts, max_norm: float, lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8,
             weight_decay=0.1, lr_schedule=None, shards=None) -> Result:
        """One attempted logical update over k micro-batches (grads[i] is a flat
        array of P gradient values: uint16 bits for bf16/f16, float32 for f32; for
        e4m3b16 a pair (uint8 codes of P elements, float32 block scales)).  With
        lr_schedule (float32 rates of optimizer steps 1, 2, ...) the rate is the
        schedule's entry for the step this update would commit, in place of lr.
        shards=(nranks, align): the sharded statement of the same update (every rank's
        slice simulated in turn, flags and squared norms combined across ranks); the
        per-rank squared norms and flags are left in self.rank_sumsq / self.rank_flag."""
        if lr_schedule is not None:
            table = np.ascontiguousarray(lr_schedule, dtype=np.float32)
            assert table.size > 0
            lr = self.lib.tlo_scheduled_lr(_ptr(table), table.size, self.state.t)
        k = len(grads)
        if self.gdtype == DT_E4M3B16:
            assert self.numel is not None and int(self.numel.sum()) == self.P
            keep = []
            for codes, scales in grads:
                c = np.ascontiguousarray(codes, dtype=np.uint8)
                sc = np.ascontiguousarray(scales, dtype=np.float32)
                assert c.size == self.P and sc.size == int(((self.numel + 15) // 16).sum())
                keep.append((c, sc, E4M3List(c.ctypes.data, sc.ctypes.data, self.numel.ctypes.data,
                                              self.numel.size)))
            gptrs = (ctypes.c_void_p * k)(*[ctypes.addressof(x[2]) for x in keep])
        else:
            gs = [np.ascontiguousarray(g) for g in grads]
            for g in gs:
                assert g.size == self.P
            gptrs = (ctypes.c_void_p * k)(*[g.ctypes.data for g in gs])
        cnts = (ctypes.c_int64 * k)(*[int(c) for c in counts])
        hp = AdamWHP(lr, beta1, beta2, eps, weight_decay)
        res = Result()
        args = (_ptr(self.w), _ptr(self.m), _ptr(self.v), _ptr(self.p), self.pdtype, _ptr(self.acc), self.P, gptrs,
                self.gdtype, cnts, k, float(max_norm), ctypes.byref(hp), ctypes.byref(self.cfg),
                ctypes.byref(self.state), ctypes.byref(res))
        if shards is None:
            rc = self.lib.tlo_step(*args)
        else:
            nranks, align = int(shards[0]), int(shards[1])
            self.rank_sumsq = np.zeros(nranks, dtype=np.float64)
            self.rank_flag = np.zeros(nranks, dtype=np.int32)
            rc = self.lib.tlo_step_sharded(*args, nranks, align, _ptr(self.rank_sumsq), _ptr(self.rank_flag))
        if rc != 0:
            raise ValueError("oracle rejected the logical update (counts must be positive, N <= 2^53)")
        self.last = res
        return res

    def scalars(self) -> dict:
        s = self.state
        return {"S": s.S, "count": s.count, "t": s.t, "b1p": s.b1p, "b2p": s.b2p}


# ---- element-wise helpers over numpy arrays (loops in C) -------------------

def partition_bounds(P: int, nranks: int, align: int = 1) -> np.ndarray:
    """Cut points of the sharded statement: slice r is [b[r], b[r+1])."""
    b = np.zeros(nranks + 1, dtype=np.int64)
    load().tlo_partition_bounds(int(P), int(nranks), int(align), _ptr(b))
    return b


def recast(x: np.ndarray, dtype: str) -> np.ndarray:
    """rd16: fp32 -> bf16/f16 bits, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    load().tlo_recast(_ptr(x), _ptr(out), x.size, _DT_BY_NAME[dtype])
    return out


def decode16(bits: np.ndarray, dtype: str) -> np.ndarray:
    """bf16/f16 bits -> fp32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(bits.size, dtype=np.float32)
    load().tlo_decode16(_ptr(bits), _ptr(out), bits.size, _DT_BY_NAME[dtype])
    return out


def e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes -> fp32 (exact)."""
    lib = load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.tlo_e4m3_to_f32(int(c)) for c in codes], dtype=np.float32)


def dequant_e4m3b16(codes: np.ndarray, scales: np.ndarray, numel) -> np.ndarray:
    """8-bit gradients of a tensor list -> fp32 values code * block scale."""
    c = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    sc = np.ascontiguousarray(scales, dtype=np.float32).ravel()
    n = np.ascontiguousarray(numel, dtype=np.int64)
    out = np.empty(c.size, dtype=np.float32)
    lst = E4M3List(c.ctypes.data, sc.ctypes.data, n.ctypes.data, n.size)
    load().tlo_dequant_e4m3b16(ctypes.byref(lst), _ptr(out))
    return out
