"""Test harness: the same seeded inputs through the GPU library and through the oracle.

GPU side: the tensor lists live in flat device buffers (optionally with seeded
0-3 element gaps before every tensor, so many tensors start off a 16-byte
boundary), and the library is driven through the Python binding of its C ABI.
Oracle side: flat numpy arrays in tensor order.  Comparisons count units in the
last place as the distance between ordered bit patterns.
"""
from __future__ import annotations

import numpy as np

import loss_scaled_adamw_gb300 as tl
from loss_scaled_adamw_gb300 import workloads as W

DT = {"bf16": tl.TL_BF16, "f16": tl.TL_F16, "f32": tl.TL_F32, "e4m3b16": tl.TL_E4M3B16}


def ordered32(a: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.int64)
    return np.where(b & 0x80000000, -(b & 0x7FFFFFFF), b)


def ordered16(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_distance32(x, y) -> np.ndarray:
    return np.abs(ordered32(x) - ordered32(y))


def ulp_distance16(x, y) -> np.ndarray:
    return np.abs(ordered16(x) - ordered16(y))


def assert_ulps32(gpu, ref, max_ulps: int, what: str):
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    assert gpu.shape == ref.shape, what
    nan_g, nan_r = np.isnan(gpu), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    d = ulp_distance32(gpu[~nan_r], ref[~nan_r])
    worst = int(d.max()) if d.size else 0
    assert worst <= max_ulps, f"{what}: {int((d > max_ulps).sum())} elements beyond {max_ulps} ulp (worst {worst})"
    return {"max_ulps": worst, "exact_fraction": float((d == 0).mean()) if d.size else 1.0}


def assert_ulps16(gpu_bits, ref_bits, max_ulps: int, what: str):
    g = np.asarray(gpu_bits).view(np.uint16)
    r = np.asarray(ref_bits).view(np.uint16)
    d = ulp_distance16(g, r)
    worst = int(d.max()) if d.size else 0
    assert worst <= max_ulps, f"{what}: {int((d > max_ulps).sum())} elements beyond {max_ulps} ulp (worst {worst})"
    return {"max_ulps": worst, "exact_fraction": float((d == 0).mean()) if d.size else 1.0}


def build_index(numel, offs, device):
    """Device index map from flat tensor-order position to buffer position."""
    import torch
    n = torch.tensor(numel, dtype=torch.int64)
    shift = torch.tensor(offs, dtype=torch.int64) - (torch.cumsum(n, 0) - n)
    return torch.arange(int(n.sum()), dtype=torch.int64, device=device) + torch.repeat_interleave(
        shift.to(device), n.to(device))


class DeviceList:
    """One tensor list in a flat device buffer; `ptrs` are the tensors' addresses."""

    def __init__(self, numel, dtype, gaps, key: int, device="cuda", fill=0.0):
        """gaps: False (every tensor on a 32-byte boundary), True (seeded 0-3 element gaps,
        independent per list) or "packed" (back to back, no padding: every list puts a
        tensor at the same element offset)."""
        import torch
        self.numel = list(numel)
        if gaps == "packed":
            self.offs, total = W.layout_offsets(self.numel, False, 1, key)
        else:
            self.offs, total = W.layout_offsets(self.numel, bool(gaps), 8, key)
        self.torch_dtype = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
        self.buf = torch.full((total + 16,), fill, dtype=self.torch_dtype, device=device)
        packed = self.offs == list(np.cumsum([0] + self.numel[:-1])) if self.numel else True
        # a packed layout needs no index map: buffer position = tensor-order position
        self.index = None if packed else build_index(self.numel, self.offs, device)
        self.P = int(sum(self.numel))
        es = self.buf.element_size()
        base = self.buf.data_ptr()
        self.ptrs = tl.PtrList([base + o * es for o in self.offs])
        self.ptrs.keep = self.buf  # keep the buffer alive with the pointer array

    def load(self, flat):
        if self.index is None:
            self.buf[:self.P].copy_(flat)
        else:
            self.buf[self.index] = flat.to(self.buf.device, self.torch_dtype)

    def flat(self):
        if self.index is None:
            return self.buf[:self.P]
        return self.buf[self.index]


class E4M3DeviceList:
    """One list of 8-bit gradient tensors in a flat device buffer: each tensor starts on a
    16-byte boundary and holds its E4M3 codes (padded to 16 bytes) and then its fp32 block
    scales; gaps=True puts a seeded 0-3 x 16 byte gap before every tensor."""

    def __init__(self, numel, gaps, key: int, device="cuda"):
        import torch
        self.numel = list(numel)
        offs, soffs, total = W.e4m3_layout(self.numel, bool(gaps), key)
        self.buf = torch.full((total + 16,), 0xEE, dtype=torch.uint8, device=device)
        n = torch.tensor(self.numel, dtype=torch.int64)
        nb = (n + 15) // 16
        P, NB = int(n.sum()), int(nb.sum())
        self.code_index = (torch.arange(P, dtype=torch.int64) + torch.repeat_interleave(
            torch.tensor(offs, dtype=torch.int64) - (torch.cumsum(n, 0) - n), n)).to(device)
        # scale b of tensor t sits at byte soffs[t] + 4 b, i.e. float index soffs[t] / 4 + b
        self.scale_index = (torch.arange(NB, dtype=torch.int64) + torch.repeat_interleave(
            torch.tensor(soffs, dtype=torch.int64) // 4 - (torch.cumsum(nb, 0) - nb), nb)).to(device)
        base = self.buf.data_ptr()
        self.ptrs = tl.PtrList([base + o for o in offs])
        self.ptrs.keep = self.buf

    def load(self, pair):
        import torch
        codes, scales = pair
        self.buf[self.code_index] = codes.to(self.buf.device)
        self.buf.view(torch.float32)[self.scale_index] = scales.to(self.buf.device)


class GpuOptimizer:
    """The GPU library over one workload's tensor list."""

    def __init__(self, wl: W.Workload, master0, gaps=False, device="cuda", key=0):
        import torch
        self.wl = wl
        self.gaps = gaps
        self.device = device
        self.key = key
        self.lists = {
            "param": DeviceList(wl.numel, wl.param_dtype, gaps, 10 + key, device),
            "master": DeviceList(wl.numel, "f32", gaps, 11 + key, device),
            "m": DeviceList(wl.numel, "f32", gaps, 12 + key, device),
            "v": DeviceList(wl.numel, "f32", gaps, 13 + key, device),
            # acc starts as garbage: the first micro-batch must overwrite it
            "acc": DeviceList(wl.numel, "f32", gaps, 14 + key, device, fill=1.0e30),
        }
        self.lists["master"].load(master0)
        self.lists["param"].load(W.to_16bit(master0.to(device), wl.param_dtype))
        cfg = tl.make_config(DT[wl.param_dtype], DT[wl.grad_dtype], wl.scaler_enabled, wl.init_scale
                             if wl.scaler_enabled else 1.0, interval=wl.interval, min_scale=wl.min_scale,
                             max_scale=wl.max_scale)
        L = self.lists
        self.ctx = tl.tl_create(wl.numel, L["param"].ptrs, L["master"].ptrs, L["m"].ptrs, L["v"].ptrs,
                                L["acc"].ptrs, cfg)
        self.grad_lists = {}

    def grad_list(self, slot: int, flat):
        """Place a flat gradient tensor into the device grad list `slot`."""
        if slot not in self.grad_lists:
            if self.wl.grad_dtype == "e4m3b16":
                self.grad_lists[slot] = E4M3DeviceList(self.wl.numel, self.gaps, 100 + slot + self.key, self.device)
            else:
                self.grad_lists[slot] = DeviceList(self.wl.numel, self.wl.grad_dtype, self.gaps,
                                                   100 + slot + self.key, self.device)
        self.grad_lists[slot].load(flat)
        return self.grad_lists[slot].ptrs

    def step(self, grads_flat, counts, hp=None, max_norm=None, resident=False):
        hp = hp or W.HP
        mbs = [self.grad_list(i, g) for i, g in enumerate(grads_flat)]
        tl.logical_update(self.ctx, mbs, counts, self.wl.max_norm if max_norm is None else max_norm,
                          tl.tl_adamw_hp(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"]),
                          resident=resident)

    def status(self):
        return tl.tl_read_status(self.ctx)

    def pull(self):
        import torch
        torch.cuda.synchronize()
        out = {}
        for k in ("master", "m", "v"):
            out[k] = self.lists[k].flat().cpu().numpy()
        out["param"] = self.lists["param"].flat().cpu().view(torch.int16).numpy().view(np.uint16)
        return out


def oracle_for(wl: W.Workload, master0):
    import oracle
    import torch
    p0 = W.to_16bit(master0.cpu(), wl.param_dtype).view(torch.int16).numpy().view(np.uint16)
    return oracle.Oracle(master0.cpu().numpy().astype(np.float32), p0, param_dtype=wl.param_dtype,
                         grad_dtype=wl.grad_dtype, scaler_enabled=wl.scaler_enabled,
                         init_scale=wl.init_scale, interval=wl.interval, min_scale=wl.min_scale,
                         max_scale=wl.max_scale, numel=wl.numel)


def grad_bits(g):
    """numpy view of a gradient tensor for the oracle (uint16 bits or float32; for 8-bit
    gradients the pair of codes and block scales)."""
    import torch
    if isinstance(g, tuple):
        return g[0].cpu().numpy(), g[1].cpu().numpy()
    g = g.cpu()
    if g.dtype == torch.float32:
        return g.numpy()
    return g.view(torch.int16).numpy().view(np.uint16)


def compare_state(gpu: dict, orc, wl: W.Workload, what: str):
    stats = {}
    stats["master"] = assert_ulps32(gpu["master"], orc.w, 2, f"{what} master")
    stats["m"] = assert_ulps32(gpu["m"], orc.m, 2, f"{what} m")
    stats["v"] = assert_ulps32(gpu["v"], orc.v, 2, f"{what} v")
    stats["param"] = assert_ulps16(gpu["param"], orc.p, 1, f"{what} param")
    return stats


def compare_scalars(st, orc, res, what: str, check_norm=True):
    assert st.S == orc.state.S, f"{what}: S {st.S} vs {orc.state.S}"
    assert st.count == orc.state.count, f"{what}: count {st.count} vs {orc.state.count}"
    assert st.t == orc.state.t, f"{what}: t {st.t} vs {orc.state.t}"
    assert st.skipped == res.skipped, f"{what}: skipped {st.skipped} vs {res.skipped}"
    assert st.b1p == orc.state.b1p and st.b2p == orc.state.b2p, f"{what}: beta powers"
    if check_norm and not res.skipped:
        assert abs(st.norm - res.norm) <= 1e-6 * abs(res.norm), f"{what}: norm {st.norm} vs {res.norm}"
        assert abs(st.coef - res.coef) <= 2e-6 * abs(res.coef), f"{what}: coef {st.coef} vs {res.coef}"


def run_parity(wl: W.Workload, gaps=False, device="cuda", steps=None, compare_every=1, hp=None, max_norm=None,
               resident=False, lr_schedule=None):
    """Run `steps` logical updates of a workload on the GPU and in the oracle from the same
    inputs, comparing scalars after every step and the state every `compare_every` steps.
    resident=True drives the many-list pass (all k micro-batches read in one pass).
    lr_schedule (float32 rates of optimizer steps 1, 2, ...) is set on the device and
    given to the oracle."""
    import torch
    master0 = W.master_init(wl, "cpu")
    gpu = GpuOptimizer(wl, master0, gaps=gaps, device=device)
    orc = oracle_for(wl, master0)
    hp = hp or W.HP
    mn = wl.max_norm if max_norm is None else max_norm
    steps = wl.steps if steps is None else steps
    okw = {}
    if lr_schedule is not None:
        table = np.ascontiguousarray(lr_schedule, dtype=np.float32)
        tl.tl_set_lr_schedule(gpu.ctx, torch.from_numpy(table).to(device))
        okw["lr_schedule"] = table
    log = []
    for step in range(1, steps + 1):
        counts = wl.counts(step)
        S = orc.state.S  # the oracle's loss scale decides how the next gradients are scaled
        grads = [W.grad_input(wl, step, i, scale=S, device="cpu") for i in range(wl.k)]
        gpu.step(grads, counts, hp=hp, max_norm=mn, resident=resident)
        res = orc.step([grad_bits(g) for g in grads], counts, mn, **hp, **okw)
        st = gpu.status()
        compare_scalars(st, orc, res, f"{wl.name} step {step}")
        entry = {"step": step, "skipped": res.skipped, "S": st.S, "norm_gpu": st.norm, "norm_oracle": res.norm}
        if step % compare_every == 0 or step == steps:
            entry["state"] = compare_state(gpu.pull(), orc, wl, f"{wl.name} step {step}")
        log.append(entry)
    return gpu, orc, log


# ---------------------------------------------------------------------------
# the oracle over very long lists: element-wise oracle functions called on disjoint
# contiguous slices from several threads (ctypes releases the GIL during a foreign
# call).  Each element still goes through the oracle's own arithmetic; nothing here
# adds, reorders or fuses an operation.  Sums keep the oracle's sequential order.
# ---------------------------------------------------------------------------

def host_threads() -> int:
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _slices(P: int, parts: int):
    step = (P + parts - 1) // parts
    return [(lo, min(P, lo + step)) for lo in range(0, P, max(step, 1))]


def parallel_slices(fn, P: int, threads: int = 0):
    """Run fn(lo, hi) over disjoint contiguous slices of [0, P) on host threads; returns
    the per-slice results in slice order."""
    from concurrent.futures import ThreadPoolExecutor
    threads = threads or host_threads()
    sl = _slices(P, threads)
    if len(sl) <= 1:
        return [fn(lo, hi) for lo, hi in sl]
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda s: fn(*s), sl))


def oracle_accumulate_par(lib, acc, vals, dt: int, w: float, first: bool):
    """The oracle's accumulate (acc = w*g, or fma(w, g, acc)) over a long flat list."""
    import ctypes
    es = vals.dtype.itemsize
    a0, g0 = acc.ctypes.data, vals.ctypes.data
    parallel_slices(lambda lo, hi: lib.tlo_accumulate(ctypes.c_void_p(a0 + 4 * lo), ctypes.c_void_p(g0 + es * lo),
                                                      dt, hi - lo, w, 1 if first else 0), acc.size)


def oracle_unscale_par(lib, acc, S: float) -> int:
    """The oracle's unscale and finite check over a long flat list (the flag is the OR of
    the slices' flags)."""
    import ctypes
    a0 = acc.ctypes.data
    return int(any(parallel_slices(lambda lo, hi: lib.tlo_unscale_check(ctypes.c_void_p(a0 + 4 * lo), hi - lo, S),
                                   acc.size)))


def oracle_dequant_par(codes, scales, numel):
    """The oracle's 8-bit dequantization of a whole tensor list, tensor ranges on threads
    (each range's codes and block scales are contiguous in tensor order)."""
    import ctypes
    import oracle
    lib = oracle.load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    n = np.ascontiguousarray(numel, dtype=np.int64)
    out = np.empty(codes.size, dtype=np.float32)
    ce = np.concatenate([[0], np.cumsum(n)])
    se = np.concatenate([[0], np.cumsum((n + 15) // 16)])
    # tensor ranges of about equal element counts
    parts = host_threads()
    bounds = sorted(set([0, n.size] + [int(np.searchsorted(ce, ce[-1] * i / parts)) for i in range(1, parts)]))

    def one(i):
        t0, t1 = bounds[i], bounds[i + 1]
        if t1 <= t0:
            return
        lst = oracle.E4M3List(codes.ctypes.data + int(ce[t0]), scales.ctypes.data + 4 * int(se[t0]),
                              n.ctypes.data + 8 * t0, t1 - t0)
        lib.tlo_dequant_e4m3b16(ctypes.byref(lst), ctypes.c_void_p(out.ctypes.data + 4 * int(ce[t0])))

    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(parts) as ex:
        list(ex.map(one, range(len(bounds) - 1)))
    return out
