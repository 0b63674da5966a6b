"""Seeded synthetic workloads of the optimizer step (shapes, distributions, seeds).

This module holds no arithmetic of the method: it only decides tensor-list
shapes, target counts and the random inputs (initial master weights, micro-batch
gradients, injected inf/NaN), so that the GPU library and the CPU oracle are fed
identical inputs.  Nothing here is produced by the GPU library.

Workloads (all seeded with 39):
  bf16_small      12 tensors x 4,096; k=2 micro-batches with 6 and 3 valid targets
                  (the Rust chapter's 9-target fixture); grads N(0, 1e-2) bf16; 3 steps;
                  no loss scaling; clip 1.0 (the expected norm ~1.65 makes it clip).
  fp16_scaled     64 x 16,384; k=1; unscaled grads N(0, 1e-6) fed as fp16(S*g) at the
                  current S; S0=2^16, growth x2 every 4 clean steps; +inf at step 3,
                  NaN (0x7E00) at step 11; 20 steps.
  llama_10m       the ~10.3M-parameter Llama tensor list (d=288, 8 layers, ffn 768, tied
                  8192-row embedding, 74 tensors); k=4 micro-batches of 8x512 positions
                  with 5-20% padding; grads N(0, 1e-2) bf16; 10 steps.
  llama_1b        the ~1.24B-parameter Llama tensor list (d=2048, 16 layers, ffn 8192,
                  q/o 2048x2048, k/v 2048x512, tied 128,256-row embedding, 146 tensors);
                  k=8; grads N(0, 1e-3) bf16; 5 timed steps.
  ragged_100k     100,000 tensors with lognormal sizes (median 512, max 2^20, ~400M total);
                  fp16 params and grads, grads N(0, 1e-2) * S with S = 2^14; k=2; inf in
                  one element of micro-batch 1 at step 2; 3 steps.
  ragged_25k      25,000 tensors of the ragged list's size distribution (~100M parameters), as
                  ragged_100k without the injected inf: a small case for counter captures.
  stream_64m      16 x 4M = 64M parameters, bf16, k=3: a small case of the same kernels for
                  hardware-counter captures (each list larger than L2).
  fp8_small       8-bit gradients ("Training at Scale" section 41.5: E4M3 codes with one fp32
                  scale per block of 16): 10 tensors (4,096 x 6 and 1, 17, 1,000, 33,333), bf16
                  params, k=3, grads N(0, 1e-2), a NaN code in micro-batch 2 of step 3; 4 steps.
  llama_1b_fp8    the llama_1b tensor list and counts with 8-bit block-scaled gradients.
  stream_64m_fp8  stream_64m's list with 8-bit gradients and k=8 (counter captures).
Every workload uses AdamW lr 1e-3, betas (0.9, 0.95), eps 1e-8, weight decay 0.1 and
master weights N(0, 0.02).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np

SEED = 39
HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


@dataclasses.dataclass
class Workload:
    name: str
    numel: List[int]
    param_dtype: str          # "bf16" | "f16"
    grad_dtype: str           # "bf16" | "f16" | "f32" | "e4m3b16"
    steps: int
    k: int
    grad_std: float
    scaler_enabled: bool = False
    init_scale: float = 1.0
    interval: int = 2000
    min_scale: float = 1.0            # the loss scale's floor and cap (powers of two)
    max_scale: float = 2.0 ** 127
    max_norm: float = 1.0
    master_std: float = 0.02
    # (step, micro-batch) -> list of (flat element index, 16-bit pattern)
    injections: Dict[Tuple[int, int], List[Tuple[int, int]]] = dataclasses.field(default_factory=dict)
    fixed_counts: Optional[List[int]] = None
    grads_prescaled: bool = False   # gradients are fed as 16-bit(S * g) at the current S

    @property
    def P(self) -> int:
        return int(sum(self.numel))

    def counts(self, step: int) -> List[int]:
        """Valid targets of the k micro-batches of a step (8x512 positions, 5-20% padding)."""
        if self.fixed_counts is not None:
            return list(self.fixed_counts)
        rng = np.random.default_rng([SEED, 7, step])
        p = rng.uniform(0.05, 0.20, self.k)
        return [int(round(4096 * (1.0 - x))) for x in p]


def llama_numel(d: int, layers: int, ffn: int, vocab: int, kv: int) -> List[int]:
    """Tensor list of a Llama decoder with a tied embedding: embedding first, then per
    layer wq, wk, wv, wo, w1 (gate), w3 (up), w2 (down), attention and MLP RMSNorm
    weights, then the final norm."""
    out = [vocab * d]
    for _ in range(layers):
        out += [d * d, kv * d, kv * d, d * d, ffn * d, ffn * d, d * ffn, d, d]
    out.append(d)
    return out


def ragged_numel(n: int = 100_000, median: int = 512, max_size: int = 1 << 20,
                 target_total: int = 400_000_000) -> List[int]:
    """Lognormal sizes clamp(round(exp(ln median + sigma z)), 1, max); sigma is solved by
    bisection (for these seeded z) so the total comes close to target_total."""
    z = np.random.default_rng([SEED, 4]).standard_normal(n)

    def sizes(sigma):
        return np.clip(np.rint(np.exp(math.log(median) + sigma * z)), 1, max_size).astype(np.int64)

    lo, hi = 0.5, 4.0
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if sizes(mid).sum() < target_total:
            lo = mid
        else:
            hi = mid
    return [int(x) for x in sizes(0.5 * (lo + hi))]


def make(name: str) -> Workload:
    if name == "bf16_small":
        return Workload(name, [4096] * 12, "bf16", "bf16", steps=3, k=2, grad_std=1e-2, fixed_counts=[6, 3])
    if name == "fp16_scaled":
        return Workload(name, [16384] * 64, "f16", "f16", steps=20, k=1, grad_std=1e-6, scaler_enabled=True,
                        init_scale=2.0 ** 16, interval=4, fixed_counts=[4096], grads_prescaled=True,
                        injections={(3, 0): [(123_457, 0x7C00)], (11, 0): [(777_777, 0x7E00)]})
    if name == "llama_10m":
        return Workload(name, llama_numel(288, 8, 768, 8192, 288), "bf16", "bf16", steps=10, k=4, grad_std=1e-2)
    if name == "llama_1b":
        return Workload(name, llama_numel(2048, 16, 8192, 128256, 512), "bf16", "bf16", steps=5, k=8,
                        grad_std=1e-3)
    if name == "ragged_100k":
        nm = ragged_numel()
        return Workload(name, nm, "f16", "f16", steps=3, k=2, grad_std=1e-2, scaler_enabled=True,
                        init_scale=2.0 ** 14, interval=2000, grads_prescaled=True,
                        injections={(2, 0): [(int(sum(nm) * 0.61803), 0x7C00)]})
    if name == "fp8_small":
        return Workload(name, [4096] * 6 + [1, 17, 1000, 33333], "bf16", "e4m3b16", steps=4, k=3, grad_std=1e-2,
                        injections={(3, 1): [(4096 * 6 + 500, 0x7F)]})
    if name == "llama_1b_fp8":
        return Workload(name, llama_numel(2048, 16, 8192, 128256, 512), "bf16", "e4m3b16", steps=5, k=8,
                        grad_std=1e-3)
    if name == "stream_64m_fp8":
        # the same small case with 8-bit gradients, k = 8 (lists of 80 MB each)
        return Workload(name, [1 << 22] * 16, "bf16", "e4m3b16", steps=2, k=8, grad_std=1e-3)
    if name == "ragged_25k":
        # a small case of the ragged list's kernels for counter captures: 25,000 tensors of
        # the same size distribution, ~100M parameters (about 2.2 GB of device memory)
        nm = ragged_numel(25_000, target_total=100_000_000)
        return Workload(name, nm, "f16", "f16", steps=3, k=2, grad_std=1e-2, scaler_enabled=True,
                        init_scale=2.0 ** 14, interval=2000, grads_prescaled=True)
    if name == "stream_64m":
        # a small case of the 1.24B workload's kernels for counter captures: every list
        # is larger than the 129 MB L2 while the whole case holds ~1.5 GB of HBM
        return Workload(name, [1 << 22] * 16, "bf16", "bf16", steps=2, k=3, grad_std=1e-3)
    raise KeyError(name)


NAMES = ("bf16_small", "fp16_scaled", "llama_10m", "llama_1b", "ragged_100k", "fp8_small", "llama_1b_fp8")


# ---------------------------------------------------------------------------
# Random inputs (torch generators; identical tensors go to the GPU and the oracle)
# ---------------------------------------------------------------------------

def _gen(device, *key: int):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([SEED, *key]).generate_state(1, np.uint64)[0] & ((1 << 63) - 1)))
    return g


def master_init(wl: Workload, device="cpu"):
    """Flat fp32 master weights N(0, master_std) over the whole tensor list."""
    import torch
    return torch.randn(wl.P, generator=_gen(device, 1), device=device, dtype=torch.float32) * wl.master_std


def to_16bit(x, dtype: str):
    """fp32 tensor -> bf16/f16 tensor (torch's round-to-nearest-even cast)."""
    import torch
    return x.to(torch.bfloat16 if dtype == "bf16" else torch.float16)


def grad_fp32(wl: Workload, step: int, mb: int, device="cpu", lo: int = 0, hi: Optional[int] = None):
    """Unscaled micro-batch gradient (fp32, flat): N(0, grad_std)."""
    import torch
    hi = wl.P if hi is None else hi
    g = torch.randn(wl.P, generator=_gen(device, 2, step, mb), device=device, dtype=torch.float32)
    return g[lo:hi] * wl.grad_std if (lo, hi) != (0, wl.P) else g * wl.grad_std


def grad_input(wl: Workload, step: int, mb: int, scale: float = 1.0, device="cpu"):
    """The gradient handed to the optimizer for micro-batch mb of step (1-based step):
    the gradient of the micro-batch mean loss times S, in grad_dtype, with the workload's
    inf/NaN injections applied.  For e4m3b16 a pair (uint8 codes of the whole list in
    tensor order, fp32 block scales of every tensor in tensor order)."""
    import torch
    g = grad_fp32(wl, step, mb, device)
    if wl.grads_prescaled:
        g = g * float(scale)      # S is a power of two: exact in fp32
    if wl.grad_dtype == "e4m3b16":
        codes, scales = quantize_e4m3b16(g, wl.numel)
        for idx, bits in wl.injections.get((step, mb), []):
            codes[idx] = bits
        return codes, scales
    if wl.grad_dtype == "f32":
        out = g
    else:
        out = to_16bit(g, wl.grad_dtype)
    for idx, bits in wl.injections.get((step, mb), []):
        if wl.grad_dtype == "f32":
            out[idx] = float("inf") if bits == 0x7C00 else float("nan")
        else:
            out.view(torch.int16)[idx] = np.int16(np.uint16(bits).view(np.int16)).item()
    return out


def quantize_e4m3b16(x, numel: List[int]):
    """What a producer of 8-bit gradients hands over ("Training at Scale" section 41.5
    recipe): per tensor, blocks of 16 consecutive elements (the last one may be short),
    scale = max |x| over the block / 448 (1 for an all-zero block), codes = E4M3 of
    x / scale rounded to nearest even (torch's float8_e4m3fn cast).  Returns (uint8 codes,
    P elements; fp32 scales, every tensor's blocks in tensor order)."""
    import torch
    dev = x.device
    n = torch.tensor(numel, dtype=torch.int64, device=dev)
    nb = (n + 15) // 16
    start = torch.cumsum(n, 0) - n
    pstart = (torch.cumsum(nb, 0) - nb) * 16
    P = int(n.sum())
    # position of every element in a layout where each tensor is padded to whole blocks
    pos = torch.arange(P, dtype=torch.int64, device=dev) + torch.repeat_interleave(pstart - start, n)
    padded = torch.zeros(int(nb.sum()) * 16, dtype=torch.float32, device=dev)
    padded[pos] = x.float()
    blocks = padded.view(-1, 16)
    scale = blocks.abs().amax(dim=1) / 448.0
    scale = torch.where(scale == 0, torch.ones_like(scale), scale)
    codes = (blocks / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1)[pos]
    return codes.contiguous(), scale.contiguous()


def e4m3_layout(numel: List[int], gaps: bool, seed_key: int) -> Tuple[List[int], List[int], int]:
    """Byte offsets of each 8-bit gradient tensor in one flat buffer: every tensor starts on
    a 16-byte boundary (with gaps, after a seeded 0-3 x 16 byte gap) and holds its codes
    padded to 16 bytes, then its block scales.  Returns (tensor offsets, scale offsets,
    total bytes)."""
    rng = np.random.default_rng([SEED, 6, seed_key])
    gap = rng.integers(0, 4, len(numel)) if gaps else np.zeros(len(numel), np.int64)
    offs, soffs, pos = [], [], 0
    for n, g in zip(numel, gap):
        pos += 16 * int(g)
        nb = (int(n) + 15) // 16
        offs.append(pos)
        soffs.append(pos + 16 * nb)
        pos = (pos + 20 * nb + 15) // 16 * 16
    return offs, soffs, pos


def layout_offsets(numel: List[int], gaps: bool, align_elems: int, seed_key: int) -> Tuple[List[int], int]:
    """Element offsets of each tensor inside one flat buffer.  Without gaps tensors are
    packed back to back, each start rounded up to align_elems; with gaps a seeded 0-3
    element gap precedes every tensor, so many tensors start off any 16-byte boundary."""
    rng = np.random.default_rng([SEED, 5, seed_key])
    offs, pos = [], 0
    gap = rng.integers(0, 4, len(numel)) if gaps else np.zeros(len(numel), np.int64)
    for n, g in zip(numel, gap):
        pos += int(g)
        if not gaps and align_elems > 1:
            pos = (pos + align_elems - 1) // align_elems * align_elems
        offs.append(pos)
        pos += int(n)
    return offs, pos
