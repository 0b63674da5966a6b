"""tl_unscale_norm_noalloc, the entry point for callers that cannot call cudaMalloc
(device memory owned by another allocator, no allocation allowed after start-up, or
an allocation that would disturb a capture or memory plan).  It works from a scratch
array compiled into the library instead of memory it allocates.

Checked through the C ABI, on two calls in a row each time:
  - against the allocating entry points (tl_accumulate with one full-weight
    micro-batch, tl_unscale_check, tl_grad_norm) on the same inputs: the unscaled
    gradient bit for bit, the norm to 1e-6 relative, the clip coefficient and the
    overflow flag exactly;
  - against the oracle (its unscale/check, squared-norm sum and clip coefficient)
    with tensors 16-byte aligned, tensors at 4-byte but not 16-byte offsets (the
    scalar loop), and elements near 2^63 whose fp32 squares are finite but whose
    fp32 sums overflow (the fp64 fallback);
  - that a call after the first on a device leaves the free device memory unchanged.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import loss_scaled_adamw_gb300 as tl

pytestmark = pytest.mark.gpu

NUMEL = [1, 7, 4096, 16383, 16384, 40000, 3, 0, 129, 20000]
S = 2.0 ** 10
MAX_NORM = 1.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from loss_scaled_adamw_gb300 import _build
    _build.build()
    tl.load_library()


def _packed(numel, dtype, fill=0.0):
    """One flat buffer, each tensor starting on a 16-byte boundary; returns buffer and addresses."""
    offs, pos = [], 0
    for n in numel:
        offs.append(pos)
        pos += (n + 7) // 8 * 8
    buf = torch.full((pos + 8,), fill, dtype=dtype, device="cuda")
    es = buf.element_size()
    return buf, offs, [buf.data_ptr() + o * es for o in offs]


def _result(t):
    torch.cuda.synchronize()
    raw = t.cpu().numpy().tobytes()[: ctypes.sizeof(tl.tl_norm_result)]
    return tl.tl_norm_result.from_buffer_copy(raw)


def test_no_alloc_matches_allocating_path_twice():
    rng = np.random.default_rng(2024)
    # the allocating path: a context over the same list, gradients in fp32
    params, _, p_addr = _packed(NUMEL, torch.bfloat16)
    master, _, w_addr = _packed(NUMEL, torch.float32)
    m, _, m_addr = _packed(NUMEL, torch.float32)
    v, _, v_addr = _packed(NUMEL, torch.float32)
    acc_ref, offs, a_addr = _packed(NUMEL, torch.float32)
    grads, _, g_addr = _packed(NUMEL, torch.float32)
    cfg = tl.make_config(tl.TL_BF16, tl.TL_F32, scaler_enabled=True, init_scale=S, interval=1000)
    ctx = tl.tl_create(NUMEL, tl.PtrList(p_addr), tl.PtrList(w_addr), tl.PtrList(m_addr), tl.PtrList(v_addr),
                       tl.PtrList(a_addr), cfg)
    # the allocation-free path: its own fp32 list and a result slot
    acc_na, _, na_addr = _packed(NUMEL, torch.float32)
    out = torch.zeros(4, dtype=torch.float64, device="cuda")
    gptrs = tl.PtrList(g_addr)
    for call in range(2):
        vals = (rng.standard_normal(grads.numel()) * 0.01 * S).astype(np.float32)
        if call == 1:
            vals[offs[5] + 123] = np.inf  # the second call overflows
        grads.copy_(torch.from_numpy(vals))
        acc_na.copy_(grads)
        # allocating path: acc = 1 * g, u = acc / S, norm and coefficient
        tl.tl_accumulate(ctx, gptrs, 1, 1, 1)
        tl.tl_unscale_check(ctx, None, 0, 1)
        tl.tl_grad_norm(ctx, MAX_NORM)
        ref = tl.tl_read_status(ctx)
        tl.tl_clip_adamw_step(ctx, tl.tl_adamw_hp(1e-3, 0.9, 0.95, 1e-8, 0.1))
        tl.tl_scaler_update(ctx)
        # allocation-free path on the same values
        tl.tl_unscale_norm_noalloc(NUMEL, tl.PtrList(na_addr), S, MAX_NORM, out.data_ptr())
        got = _result(out)
        torch.cuda.synchronize()
        for n, o in zip(NUMEL, offs):
            a = acc_ref[o:o + n].cpu().numpy()
            b = acc_na[o:o + n].cpu().numpy()
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"call {call}: u differs"
        assert got.found_inf == ref.found_inf == (1 if call == 1 else 0), call
        if call == 0:
            assert abs(got.norm - ref.norm) <= 1e-6 * ref.norm, (got.norm, ref.norm)
            assert abs(got.coef - ref.coef) <= 2e-6 * ref.coef, (got.coef, ref.coef)
            assert abs(got.sumsq - ref.sumsq) <= 2e-6 * ref.sumsq
            assert ref.coef < 1.0  # the clip is active
        else:
            assert np.isinf(got.norm) and np.isinf(ref.norm) and got.coef == ref.coef


def _oracle_reference(vals, S, max_norm):
    """u, overflow flag, squared norm, norm and clip coefficient of one flat fp32 list from
    the oracle's functions (the allocation-free call computes exactly this)."""
    import oracle
    lib = oracle.load()
    u = np.ascontiguousarray(vals, dtype=np.float32).copy()
    P_ = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    found = lib.tlo_unscale_check(P_(u), u.size, S)
    sumsq = lib.tlo_sumsq(P_(u), u.size)
    norm = lib.tlo_norm_from_sumsq(sumsq)
    return u, found, sumsq, norm, lib.tlo_clip_coef(norm, max_norm)


def _place(numel, misalign):
    """Tensor offsets (in fp32 elements) in one flat buffer: 16-byte aligned, or shifted by
    1-3 elements so that most tensors start on a 4-byte but not a 16-byte boundary."""
    offs, pos = [], 0
    for i, n in enumerate(numel):
        pos = (pos + 7) // 8 * 8 + ((1 + i % 3) if misalign else 0)
        offs.append(pos)
        pos += n
    return offs, pos


@pytest.mark.parametrize("case", ["aligned", "misaligned", "large_values"])
def test_no_alloc_matches_oracle_twice(case):
    import oracle  # noqa: F401  (built by the fixture's build step)
    misalign = case == "misaligned"
    offs, total = _place(NUMEL, misalign)
    buf = torch.zeros(total + 16, dtype=torch.float32, device="cuda")
    addrs = [buf.data_ptr() + 4 * o for o in offs]
    if misalign:
        assert sum(a % 16 != 0 for a, n in zip(addrs, NUMEL) if n) >= 6
    out = torch.zeros(4, dtype=torch.float64, device="cuda")
    rng = np.random.default_rng(7 + len(case))
    free_before_second = None
    for call in range(2):
        vals = (rng.standard_normal(total) * 0.01 * S).astype(np.float32)
        if case == "large_values":
            # u near 1.5 * 2^63: each fp32 square (about 1.9e38) is finite, the sum of two is not
            for o, n in zip(offs, NUMEL):
                if n >= 64:
                    vals[o + 8:o + 24] = np.float32(1.5 * 2.0 ** 63 * S) * (1 + 0.01 * np.arange(16, dtype=np.float32))
        if call == 1 and case != "large_values":
            vals[offs[5] + 77] = np.nan                  # the second call overflows
        buf[:total].copy_(torch.from_numpy(vals))
        torch.cuda.synchronize()
        if call == 1:
            free_before_second = torch.cuda.mem_get_info()[0]
        tl.tl_unscale_norm_noalloc(NUMEL, tl.PtrList(addrs), S, MAX_NORM, out.data_ptr())
        got = _result(out)
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before_second, "the second call allocated device memory"
        flat = np.concatenate([vals[o:o + n] for o, n in zip(offs, NUMEL)])
        u_ref, found, sumsq, norm, coef = _oracle_reference(flat, S, MAX_NORM)
        res = buf.cpu().numpy()
        u_gpu = np.concatenate([res[o:o + n] for o, n in zip(offs, NUMEL)])
        # bit for bit, except that a NaN's payload is not fixed by IEEE arithmetic: NaN
        # positions must agree
        nan = np.isnan(u_ref)
        assert np.array_equal(np.isnan(u_gpu), nan), f"{case} call {call}: NaN positions differ"
        assert np.array_equal(u_gpu[~nan].view(np.uint32), u_ref[~nan].view(np.uint32)), f"{case} call {call}: u differs"
        assert got.found_inf == found, (case, call, got.found_inf, found)
        if not found:
            assert abs(got.sumsq - sumsq) <= 2e-6 * sumsq, (got.sumsq, sumsq)
            assert abs(got.norm - norm) <= 1e-6 * norm, (got.norm, norm)
            assert abs(got.coef - coef) <= 2e-6 * coef, (got.coef, coef)
        if case == "large_values":
            assert found == 0 and got.norm > 1e19 and got.coef < 1e-18


def test_no_alloc_rejects_lists_beyond_its_scratch():
    out = torch.zeros(4, dtype=torch.float64, device="cuda")
    big = [1 << 30, 1]  # 2^16 + 1 chunks of 2^14: more than the scratch holds
    with pytest.raises(tl.TLError) as ei:
        tl.tl_unscale_norm_noalloc(big, tl.PtrList([1 << 40, (1 << 40) + (1 << 33)]), S, MAX_NORM, out.data_ptr())
    assert ei.value.status == tl.TL_EINVAL
    with pytest.raises(tl.TLError) as ei:
        tl.tl_unscale_norm_noalloc([1] * 257, tl.PtrList([(1 << 40) + 64 * i for i in range(257)]), S, MAX_NORM,
                                   out.data_ptr())
    assert ei.value.status == tl.TL_EINVAL
    # S must be a normal power of two: 3 is none, and below 2^-126 the reciprocal is not finite
    for bad_s in (3.0, 2.0 ** -127, 2.0 ** -149, 0.0, float("inf")):
        with pytest.raises(tl.TLError) as ei:
            tl.tl_unscale_norm_noalloc([4], tl.PtrList([1 << 40]), bad_s, MAX_NORM, out.data_ptr())
        assert ei.value.status == tl.TL_EINVAL, bad_s
