"""GB300 loss-scaled AdamW optimizer step: Python binding of the C ABI (include/tl.h).

The binding only marshals arguments: every step of the optimizer runs in the
CUDA kernels of ``libtl_gb300.so``.  PyTorch supplies device memory and the
current stream.  There is no CPU fallback: if the library is not built, or no
CUDA device is present, the calls raise.

Functions keep the C names::

    ctx = tl_create(numel, params, masters, ms, vs, accs, cfg)
    tl_accumulate(ctx, grads_1, n_1, N, first=1)          # micro-batches 1..k-1
    tl_unscale_check(ctx, grads_k, n_k, N)                  # the last one
    tl_grad_norm(ctx, max_norm)
    tl_clip_adamw_step(ctx, hp)
    tl_scaler_update(ctx)

Tensor lists are Python sequences of tensors (or a prebuilt ``PtrList``, which
avoids rebuilding the pointer array on every call for long lists).
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtl_gb300.so")

TL_OK, TL_EINVAL, TL_ECUDA, TL_ESTATE, TL_ENOMEM = 0, 1, 2, 3, 4
TL_F32, TL_BF16, TL_F16, TL_E4M3B16 = 0, 1, 2, 3

EXPORTED = ("tl_create", "tl_destroy", "tl_accumulate", "tl_accumulate_many", "tl_unscale_check_many",
            "tl_unscale_check", "tl_grad_norm",
            "tl_clip_adamw_step", "tl_scaler_update", "tl_read_status", "tl_get_state", "tl_set_state",
            "tl_scale_ptr", "tl_num_params", "tl_num_chunks", "tl_launch_count", "tl_status_string",
            "tl_last_error", "tl_unscale_norm_noalloc", "tl_loss_seed", "tl_set_lr_schedule",
            "tl_local_sumsq", "tl_grad_norm_from", "tl_partition", "tl_plan")


class TLError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = f"{fn} failed with status {status}"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class tl_config(ctypes.Structure):
    _fields_ = [("param_dtype", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("scaler_enabled", ctypes.c_int32), ("init_scale", ctypes.c_float),
                ("growth", ctypes.c_float), ("backoff", ctypes.c_float), ("interval", ctypes.c_int32),
                ("min_scale", ctypes.c_float), ("max_scale", ctypes.c_float)]


class tl_adamw_hp(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class tl_state(ctypes.Structure):
    _fields_ = [("S", ctypes.c_float), ("count", ctypes.c_int32), ("t", ctypes.c_int64),
                ("b1p", ctypes.c_double), ("b2p", ctypes.c_double)]


class tl_status(ctypes.Structure):
    _fields_ = [("S", ctypes.c_float), ("count", ctypes.c_int32), ("t", ctypes.c_int64),
                ("skipped", ctypes.c_int32), ("found_inf", ctypes.c_int32), ("norm", ctypes.c_float),
                ("coef", ctypes.c_float), ("sumsq", ctypes.c_double), ("b1p", ctypes.c_double),
                ("b2p", ctypes.c_double)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class tl_plan_info(ctypes.Structure):
    _fields_ = [("nchunks", ctypes.c_int64), ("nbig", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("seg", ctypes.c_int64), ("nsmall", ctypes.c_int64), ("run_big", ctypes.c_int32),
                ("run_small", ctypes.c_int32), ("split_forms", ctypes.c_int32), ("fused_norm", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class tl_norm_result(ctypes.Structure):
    _fields_ = [("norm", ctypes.c_float), ("coef", ctypes.c_float), ("found_inf", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("sumsq", ctypes.c_double)]


def make_config(param_dtype: int = TL_BF16, grad_dtype: int = TL_BF16, scaler_enabled: bool = False,
                init_scale: float = 2.0 ** 16, growth: float = 2.0, backoff: float = 0.5,
                interval: int = 2000, min_scale: float = 1.0, max_scale: float = 2.0 ** 127) -> tl_config:
    """Defaults follow the mixed-precision page's DynamicLossScaler(init=2^16, growth=2,
    backoff=0.5, interval=2000)."""
    return tl_config(param_dtype, grad_dtype, 1 if scaler_enabled else 0, init_scale, growth, backoff,
                     interval, min_scale, max_scale)


_lib = None


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load libtl_gb300.so.  Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with loss_scaled_adamw_gb300._build.build() "
                          "(or __graft_entry__.build()); there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    pp = ctypes.POINTER(ctypes.c_void_p)
    sigs = {
        "tl_create": (i32, [ctypes.POINTER(vp), i64, ctypes.POINTER(i64), pp, pp, pp, pp, pp,
                            ctypes.POINTER(tl_config), vp]),
        "tl_destroy": (i32, [vp]),
        "tl_accumulate": (i32, [vp, pp, i64, i64, i32, vp]),
        "tl_accumulate_many": (i32, [vp, i32, pp, ctypes.POINTER(i64), i64, i32, vp]),
        "tl_unscale_check_many": (i32, [vp, i32, pp, ctypes.POINTER(i64), i64, vp]),
        "tl_unscale_check": (i32, [vp, pp, i64, i64, vp]),
        "tl_grad_norm": (i32, [vp, f32, vp]),
        "tl_clip_adamw_step": (i32, [vp, ctypes.POINTER(tl_adamw_hp), vp]),
        "tl_scaler_update": (i32, [vp, vp]),
        "tl_read_status": (i32, [vp, ctypes.POINTER(tl_status), vp]),
        "tl_get_state": (i32, [vp, ctypes.POINTER(tl_state), vp]),
        "tl_set_state": (i32, [vp, ctypes.POINTER(tl_state), vp]),
        "tl_scale_ptr": (vp, [vp]),
        "tl_num_params": (i64, [vp]),
        "tl_num_chunks": (i64, [vp]),
        "tl_launch_count": (i64, [vp]),
        "tl_status_string": (ctypes.c_char_p, [i32]),
        "tl_last_error": (ctypes.c_char_p, [vp]),
        "tl_unscale_norm_noalloc": (i32, [i64, ctypes.POINTER(i64), pp, f32, f32, vp, vp]),
        "tl_loss_seed": (i32, [vp, i64, i64, vp, vp]),
        "tl_set_lr_schedule": (i32, [vp, vp, i64]),
        "tl_local_sumsq": (i32, [vp, vp, vp, vp]),
        "tl_grad_norm_from": (i32, [vp, vp, vp, f32, vp]),
        "tl_partition": (i32, [i64, ctypes.POINTER(i64), ctypes.c_int32, ctypes.c_int32, i64,
                               ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64), i64,
                               ctypes.POINTER(i64)]),
        "tl_plan": (i32, [i64, ctypes.POINTER(i64), ctypes.c_int32, ctypes.POINTER(tl_plan_info)]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PtrList:
    """A tensor list as a C array of data pointers (keeps the tensors alive).
    Entries may also be plain integer addresses."""

    def __init__(self, tensors: Sequence):
        self.tensors = list(tensors)
        addrs = [t if isinstance(t, int) else t.data_ptr() for t in self.tensors]
        self.array = (ctypes.c_void_p * max(len(self.tensors), 1))(*addrs)

    def __len__(self):
        return len(self.tensors)


def _ptrs(x):
    if x is None:
        return None
    if isinstance(x, PtrList):
        return x.array
    return PtrList(x).array


def _stream(stream):
    if isinstance(stream, ctypes.c_void_p):
        return stream
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class Context:
    """Owns one tl_ctx and the tensor lists it was created over."""

    def __init__(self, handle: ctypes.c_void_p, keep):
        self.handle = handle
        self._keep = keep
        self.lr_table = None  # the learning-rate schedule tensor while one is set

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.tl_destroy(self.handle)
            self.handle = None


def _check(ctx, fn: str, rc: int):
    if rc != TL_OK:
        lib = load_library()
        detail = lib.tl_last_error(ctx.handle).decode() if ctx is not None and ctx.handle else ""
        if not detail:
            detail = lib.tl_status_string(rc).decode()
        raise TLError(fn, rc, detail)


def tl_create(numel: Sequence[int], params, masters, ms, vs, accs, cfg: tl_config, stream=None) -> Context:
    lib = load_library()
    n = len(numel)
    lists = [p if isinstance(p, PtrList) else PtrList(p) for p in (params, masters, ms, vs, accs)]
    for lst in lists:
        if len(lst) != n:
            raise ValueError("every tensor list must have len(numel) entries")
    numel_arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numel])
    h = ctypes.c_void_p()
    rc = lib.tl_create(ctypes.byref(h), n, numel_arr, *[lst.array for lst in lists], ctypes.byref(cfg),
                       _stream(stream))
    if rc != TL_OK:
        raise TLError("tl_create", rc, lib.tl_status_string(rc).decode())
    return Context(h, lists)


def tl_destroy(ctx: Context) -> None:
    if ctx.handle:
        rc = load_library().tl_destroy(ctx.handle)
        ctx.handle = None
        if rc != TL_OK:
            raise TLError("tl_destroy", rc)


def tl_accumulate(ctx: Context, grads, n_i: int, N: int, first: int, stream=None) -> None:
    _check(ctx, "tl_accumulate", load_library().tl_accumulate(ctx.handle, _ptrs(grads), int(n_i), int(N),
                                                              int(first), _stream(stream)))


class ManyLists:
    """k gradient lists flattened list-major into one C pointer array (keeps them alive)."""

    def __init__(self, lists: Sequence):
        self.lists = [l if isinstance(l, PtrList) else PtrList(l) for l in lists]
        n = len(self.lists[0]) if self.lists else 0
        flat = []
        for l in self.lists:
            if len(l) != n:
                raise ValueError("every gradient list must have the same number of tensors")
            flat.extend(l.array[i] for i in range(n))
        self.k = len(self.lists)
        self.array = (ctypes.c_void_p * max(len(flat), 1))(*flat)


def tl_accumulate_many(ctx: Context, lists, counts: Sequence[int], N: int, last: int, stream=None) -> None:
    ml = lists if isinstance(lists, ManyLists) else ManyLists(lists)
    cnt = (ctypes.c_int64 * max(ml.k, 1))(*[int(c) for c in counts])
    if len(counts) != ml.k:
        raise ValueError("one count per gradient list")
    _check(ctx, "tl_accumulate_many", load_library().tl_accumulate_many(ctx.handle, ml.k, ml.array, cnt, int(N),
                                                                        int(last), _stream(stream)))


def tl_unscale_check_many(ctx: Context, lists, counts: Sequence[int], N: int, stream=None) -> None:
    ml = lists if isinstance(lists, ManyLists) else ManyLists(lists)
    if len(counts) != ml.k:
        raise ValueError("one count per gradient list")
    cnt = (ctypes.c_int64 * max(ml.k, 1))(*[int(c) for c in counts])
    _check(ctx, "tl_unscale_check_many", load_library().tl_unscale_check_many(ctx.handle, ml.k, ml.array, cnt, int(N),
                                                                              _stream(stream)))


def tl_unscale_check(ctx: Context, grads, n_k: int, N: int, stream=None) -> None:
    _check(ctx, "tl_unscale_check", load_library().tl_unscale_check(ctx.handle, _ptrs(grads), int(n_k), int(N),
                                                                    _stream(stream)))


def tl_grad_norm(ctx: Context, max_norm: float, stream=None) -> None:
    _check(ctx, "tl_grad_norm", load_library().tl_grad_norm(ctx.handle, float(max_norm), _stream(stream)))


def tl_clip_adamw_step(ctx: Context, hp: tl_adamw_hp, stream=None) -> None:
    _check(ctx, "tl_clip_adamw_step", load_library().tl_clip_adamw_step(ctx.handle, ctypes.byref(hp),
                                                                        _stream(stream)))


def tl_scaler_update(ctx: Context, stream=None) -> None:
    _check(ctx, "tl_scaler_update", load_library().tl_scaler_update(ctx.handle, _stream(stream)))


def tl_read_status(ctx: Context, stream=None) -> tl_status:
    st = tl_status()
    _check(ctx, "tl_read_status", load_library().tl_read_status(ctx.handle, ctypes.byref(st), _stream(stream)))
    return st


def tl_get_state(ctx: Context, stream=None) -> tl_state:
    st = tl_state()
    _check(ctx, "tl_get_state", load_library().tl_get_state(ctx.handle, ctypes.byref(st), _stream(stream)))
    return st


def tl_set_state(ctx: Context, state: tl_state, stream=None) -> None:
    _check(ctx, "tl_set_state", load_library().tl_set_state(ctx.handle, ctypes.byref(state), _stream(stream)))


def tl_scale_ptr(ctx: Context) -> int:
    return int(load_library().tl_scale_ptr(ctx.handle) or 0)


def tl_loss_seed(ctx: Context, n_i: int, N: int, out_addr: int, stream=None) -> None:
    """Write S * n_i / N (fp32) to the device address out_addr on the stream."""
    _check(ctx, "tl_loss_seed", load_library().tl_loss_seed(ctx.handle, int(n_i), int(N),
                                                            ctypes.c_void_p(int(out_addr)), _stream(stream)))


def tl_set_lr_schedule(ctx: Context, table) -> None:
    """Learning rates of optimizer steps 1, 2, ... read on the device (a float32 CUDA
    tensor), or None to go back to hp.lr.  The context keeps a reference to the tensor
    while it is set."""
    if table is None:
        _check(ctx, "tl_set_lr_schedule", load_library().tl_set_lr_schedule(ctx.handle, None, 0))
        ctx.lr_table = None
        return
    import torch
    if table.dtype != torch.float32 or not table.is_contiguous() or table.dim() != 1:
        raise ValueError("the schedule is a contiguous 1-D float32 tensor")
    _check(ctx, "tl_set_lr_schedule", load_library().tl_set_lr_schedule(
        ctx.handle, ctypes.c_void_p(table.data_ptr()), int(table.numel())))
    ctx.lr_table = table


def tl_local_sumsq(ctx: Context, sumsq_addr: int, flag_addr: int, stream=None) -> None:
    """Write this context's squared norm (fp64) and overflow flag (int32) to the device
    addresses on the stream (the sharded form of tl_grad_norm, first half)."""
    _check(ctx, "tl_local_sumsq", load_library().tl_local_sumsq(ctx.handle, ctypes.c_void_p(int(sumsq_addr)),
                                                                ctypes.c_void_p(int(flag_addr)), _stream(stream)))


def tl_grad_norm_from(ctx: Context, sumsq_addr: int, flag_addr: int, max_norm: float, stream=None) -> None:
    """Take the squared norm and flag combined across shards (device addresses) as the
    update's norm and overflow decision."""
    _check(ctx, "tl_grad_norm_from", load_library().tl_grad_norm_from(
        ctx.handle, ctypes.c_void_p(int(sumsq_addr)), ctypes.c_void_p(int(flag_addr)), float(max_norm),
        _stream(stream)))


def tl_partition(numel: Sequence[int], nranks: int, rank: int, align: int = 1):
    """The pieces (tensor index, first element, length) of the slice rank `rank` of
    `nranks` owns (host only)."""
    lib = load_library()
    n = len(numel)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numel])
    cap = max(n, 1)
    t, s, l = (ctypes.c_int64 * cap)(), (ctypes.c_int64 * cap)(), (ctypes.c_int64 * cap)()
    cnt = ctypes.c_int64()
    rc = lib.tl_partition(n, arr, int(nranks), int(rank), int(align), t, s, l, cap, ctypes.byref(cnt))
    if rc != TL_OK:
        raise TLError("tl_partition", rc, lib.tl_status_string(rc).decode())
    return [(int(t[q]), int(s[q]), int(l[q])) for q in range(cnt.value)]


def tl_plan(numel: Sequence[int], sm_count: int = 152) -> dict:
    """How tl_create lays out a tensor list of these sizes on a device of sm_count SMs
    (host only): the chunk table's counts, the segment length, the squared-norm run
    lengths, whether the split forms run and whether the pass finishes the norm."""
    lib = load_library()
    n = len(numel)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numel])
    out = tl_plan_info()
    rc = lib.tl_plan(n, arr, int(sm_count), ctypes.byref(out))
    if rc != TL_OK:
        raise TLError("tl_plan", rc, lib.tl_status_string(rc).decode())
    return out.as_dict()


def tl_num_params(ctx: Context) -> int:
    return int(load_library().tl_num_params(ctx.handle))


def tl_num_chunks(ctx: Context) -> int:
    return int(load_library().tl_num_chunks(ctx.handle))


def tl_launch_count(ctx: Context) -> int:
    return int(load_library().tl_launch_count(ctx.handle))


def logical_update(ctx: Context, micro_batches, counts, max_norm: float, hp: tl_adamw_hp, stream=None,
                   resident=False) -> None:
    """One attempted logical update: the tl_* call sequence over k micro-batches
    (micro_batches[i] is a tensor list or PtrList; counts[i] its valid targets).
    resident=True reads all k lists in one pass (tl_accumulate_many); resident="remat"
    checks them without storing u (tl_unscale_check_many, k <= 4) and lets the AdamW
    pass recompute u from them.  With either, micro_batches may also be a prebuilt
    ManyLists."""
    k = micro_batches.k if isinstance(micro_batches, ManyLists) else len(micro_batches)
    if k < 1 or len(counts) != k:
        raise ValueError("need one count per micro-batch and at least one micro-batch")
    N = int(sum(int(c) for c in counts))
    s = _stream(stream)
    if resident == "remat":
        tl_unscale_check_many(ctx, micro_batches, counts, N, s)
    elif resident:
        tl_accumulate_many(ctx, micro_batches, counts, N, 1, s)
    else:
        for i in range(k - 1):
            tl_accumulate(ctx, micro_batches[i], counts[i], N, 1 if i == 0 else 0, s)
        tl_unscale_check(ctx, micro_batches[k - 1], counts[k - 1], N, s)
    tl_grad_norm(ctx, max_norm, s)
    tl_clip_adamw_step(ctx, hp, s)
    tl_scaler_update(ctx, s)


def tl_unscale_norm_noalloc(numel: Sequence[int], accs, S: float, max_norm: float, out_addr: int,
                            stream=None) -> None:
    """Unscale + overflow check + global norm + clip coefficient with no allocation (for
    callers that cannot call cudaMalloc): accs are fp32 device tensors overwritten with
    acc / S; out_addr is the device address of a tl_norm_result (24 bytes, 8-byte aligned)."""
    lib = load_library()
    n = len(numel)
    lst = accs if isinstance(accs, PtrList) else PtrList(accs)
    if len(lst) != n:
        raise ValueError("accs must have len(numel) entries")
    numel_arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numel])
    rc = lib.tl_unscale_norm_noalloc(n, numel_arr, lst.array, float(S), float(max_norm),
                                     ctypes.c_void_p(int(out_addr)), _stream(stream))
    if rc != TL_OK:
        raise TLError("tl_unscale_norm_noalloc", rc, lib.tl_status_string(rc).decode())
