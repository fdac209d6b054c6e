"""Seeded synthetic inputs shaped like the workloads of the Gemma 4 / Llama
decode geometries ("Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus
(Part 2)", section "One KV head breaks the textbook", geometry table).

This module holds no attention arithmetic. It draws Q, K and V as iid N(0, 1)
rounded to bf16, draws the per-sequence lengths, and can poison with NaN every
cache slot that does not hold one of the live positions, the way the page's
section "The test that catches what parity misses" describes. The CUDA library
never imports it; the tests, the benchmark and the oracle's callers do.

Layout of what it returns (the library's layout):
  q        bf16 [B, NH, HS]
  k_cache  bf16 [B, NKV, capacity, HS]   (head-major; position p in slot p % capacity)
  v_cache  bf16 [B, NKV, capacity, HS]
  lens     int32 [B]
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

BF16_NAN_BITS = 0x7FC0


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    NH: int
    NKV: int
    HS: int
    capacity: int
    window: int            # <= 0: no window
    lens: tuple = ()       # explicit per-sequence lengths, or () for ragged draw
    ragged_max: int = 0    # ragged: len ~ U[1, ragged_max]
    seed: int = 1000
    desc: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.HS)

    @property
    def G(self) -> int:
        return self.NH // self.NKV


# The five workloads (six with the two MQA lengths), with their sizes.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("llama_tiny", 1, 32, 8, 128, 512, 0, lens=(256,), seed=1000,
                 desc="Llama geometry tiny: B=1, 32 Q / 8 KV heads, d128, capacity 512, len 256"),
        Workload("gemma_local_ring", 1, 16, 8, 256, 1024, 1024, lens=(32768,), seed=1001,
                 desc="Gemma local sliding ring: B=1, 16 Q / 8 KV heads, d256, window = capacity = 1024, len 32768"),
        Workload("gemma_global_mqa_4k", 1, 16, 1, 512, 32768, 0, lens=(4096,), seed=1002,
                 desc="Gemma global MQA: B=1, 16 Q / 1 KV head, d512, capacity 32768, len 4096"),
        Workload("gemma_global_mqa_32k", 1, 16, 1, 512, 32768, 0, lens=(32768,), seed=1003,
                 desc="Gemma global MQA: B=1, 16 Q / 1 KV head, d512, capacity 32768, len 32768"),
        Workload("llama_ragged", 16, 32, 8, 128, 32768, 0, ragged_max=32768, seed=1004,
                 desc="Llama geometry batched ragged: B=16, 32 Q / 8 KV heads, d128, capacity 32768, len ~ U[1,32768]"),
        Workload("gemma_mqa_long", 4, 16, 1, 512, 131072, 0, lens=(131072,) * 4, seed=1005,
                 desc="Gemma global MQA long context: B=4, 16 Q / 1 KV head, d512, capacity = len = 131072"),
    ]
}


# Smaller cases of the same geometries for profiler captures (a few GB on the
# device at most, live band still larger than the 129 MB L2).
PROFILE_WORKLOADS = {
    w.name: w
    for w in [
        Workload("llama_ragged_b4", 4, 32, 8, 128, 32768, 0, ragged_max=32768, seed=1104,
                 desc="Llama geometry ragged, 4 sequences: 32 Q / 8 KV heads, d128, capacity 32768, len ~ U[1,32768]"),
        Workload("gemma_mqa_long_b1", 1, 16, 1, 512, 131072, 0, lens=(131072,), seed=1105,
                 desc="Gemma global MQA long context, 1 sequence: 16 Q / 1 KV head, d512, len 131072"),
        Workload("gemma_local_ring_b16", 16, 16, 8, 256, 1024, 1024, lens=(32768,) * 16, seed=1106,
                 desc="Gemma local sliding ring, 16 sequences: 16 Q / 8 KV heads, d256, window = capacity = 1024"),
    ]
}


def draw_lens(w: Workload) -> torch.Tensor:
    """Per-sequence lengths (int32, CPU). Ragged workloads draw U[1, ragged_max]
    from a generator seeded with the workload's seed."""
    if w.lens:
        assert len(w.lens) == w.B
        return torch.tensor(w.lens, dtype=torch.int32)
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    return torch.randint(1, w.ragged_max + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)


def _randn_bf16(shape, gen: torch.Generator, device, chunk_rows: int = 1 << 22) -> torch.Tensor:
    """iid N(0,1) rounded to bf16, drawn in chunks so no large fp32 temporary lives."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    step = max(1, chunk_rows)
    for a in range(0, n, step):
        e = min(n, a + step)
        flat[a:e] = torch.randn(e - a, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def live_slots(length: int, capacity: int, window: int) -> torch.Tensor:
    """Boolean [capacity]: True where the slot holds one of the positions of
    [max(0, len - min(window, capacity)), len) after tokens 0..len-1 were
    written at slot pos % capacity. Used only to poison the other slots."""
    keep = capacity if window <= 0 else min(window, capacity)
    lo = max(0, length - keep)
    mask = torch.zeros(capacity, dtype=torch.bool)
    if length - lo >= capacity:
        mask[:] = True
    elif length > lo:
        mask[torch.arange(lo, length, dtype=torch.int64) % capacity] = True
    return mask


def poison_dead_slots(k_cache: torch.Tensor, v_cache: torch.Tensor, lens, capacity: int, window: int) -> None:
    """Write bf16 NaN into every slot that holds no live position (in place)."""
    lens_l = [int(x) for x in (lens.tolist() if torch.is_tensor(lens) else lens)]
    nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    for b, length in enumerate(lens_l):
        dead = ~live_slots(length, capacity, window)
        if dead.any():
            idx = dead.nonzero().view(-1).to(k_cache.device)
            k_cache[b].index_fill_(1, idx, nan)
            v_cache[b].index_fill_(1, idx, nan)


def make_inputs(w: Workload, device="cpu", poison: bool = True, seed: int | None = None,
                lens: torch.Tensor | None = None):
    """Q, K cache, V cache (bf16) and lens (int32) for a workload, on `device`.

    Values are drawn by a torch generator on `device` seeded with the workload's
    seed (or `seed`); CPU and CUDA generators give different but individually
    reproducible draws. Lens always come from the CPU generator."""
    s = w.seed if seed is None else seed
    gen = torch.Generator(device=device).manual_seed(s)
    q = _randn_bf16((w.B, w.NH, w.HS), gen, device)
    k = _randn_bf16((w.B, w.NKV, w.capacity, w.HS), gen, device)
    v = _randn_bf16((w.B, w.NKV, w.capacity, w.HS), gen, device)
    ln = draw_lens(w) if lens is None else lens.to(torch.int32).cpu()
    if poison:
        poison_dead_slots(k, v, ln, w.capacity, w.window)
    return q, k, v, ln


E4M3_NAN_CODE = 0x7F
E4M3_MAX = 448.0


def quantize_e4m3(cache: torch.Tensor):
    """A cache writer's FP8 step: one fp32 scale per (sequence, KV head),
    absmax / 448 over its finite values, and the E4M3 codes of value / scale
    (round to nearest; NaN stays NaN). Returns (codes uint8 [B,NKV,cap,HS],
    scales fp32 [B,NKV])."""
    x = cache.float()
    finite = torch.isfinite(x)
    amax = torch.where(finite, x.abs(), torch.zeros_like(x)).amax(dim=(2, 3))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    codes = (x / scale[:, :, None, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def make_inputs_fp8(w: Workload, device="cpu", poison: bool = True, seed: int | None = None,
                    lens: torch.Tensor | None = None):
    """Q (bf16), an FP8 E4M3 K and V cache (uint8 codes) with per-(sequence,
    KV head) fp32 scales, and lens: the bf16 draw of make_inputs, quantized;
    slots holding no live position get the NaN code."""
    q, k, v, ln = make_inputs(w, device=device, poison=False, seed=seed, lens=lens)
    k8, ks = quantize_e4m3(k)
    v8, vs = quantize_e4m3(v)
    del k, v
    if poison:
        for b, length in enumerate(ln.tolist()):
            dead = ~live_slots(int(length), w.capacity, w.window)
            if dead.any():
                idx = dead.nonzero().view(-1).to(k8.device)
                k8[b].index_fill_(1, idx, E4M3_NAN_CODE)
                v8[b].index_fill_(1, idx, E4M3_NAN_CODE)
    return q, k8, v8, ks, vs, ln


def small(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (for scaled-down cases)."""
    return replace(w, **kw)


__all__ = ["Workload", "WORKLOADS", "PROFILE_WORKLOADS", "draw_lens", "make_inputs", "make_inputs_fp8",
           "quantize_e4m3", "live_slots", "poison_dead_slots", "small", "BF16_NAN_BITS", "E4M3_NAN_CODE"]
