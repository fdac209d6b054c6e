"""Naive full-softmax brute force for tiny decode-attention inputs (torch
float64 on the CPU). Independent of both the oracle and the CUDA library.

It does not gather a band. It unrolls the cache into the whole history of
positions [0, len) (position p read from slot p % capacity; positions the
cache no longer holds get zero rows), scores every one of them, masks the
positions older than the window with -inf, and applies a full softmax - the
masked-softmax formulation the old five-launch pipeline used ("Hand-Writing
Gemma 4 Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section "The starting
point"). A second routine asks torch's scaled_dot_product_attention (float64,
CPU, boolean mask, K/V heads repeated per group) for the same numbers.
"""

from __future__ import annotations

import torch
import torch.nn.functional as F


def _history(cache_b: torch.Tensor, length: int, capacity: int, keep: torch.Tensor) -> torch.Tensor:
    """[NKV, len, HS] float64: row p = cache[:, p % capacity] if the cache still
    holds position p (p >= len - capacity) and the mask keeps it, else zeros
    (a masked row gets weight exactly 0, so its content must not matter; a
    poisoned NaN there would otherwise turn 0 * NaN into NaN)."""
    pos = torch.arange(length)
    h = cache_b[:, pos % capacity, :].to(torch.float64).clone()
    gone = (pos < length - capacity) | ~keep
    h[:, gone, :] = 0.0
    return h


def _mask(length: int, window: int) -> torch.Tensor:
    pos = torch.arange(length)
    if window <= 0:
        return torch.ones(length, dtype=torch.bool)
    return pos >= length - window


def brute_force(q, k, v, lens, B, NH, NKV, HS, capacity, window, scale) -> torch.Tensor:
    """Full masked softmax over every position of the history."""
    G = NH // NKV
    out = torch.zeros(B, NH, HS, dtype=torch.float64)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        keep = _mask(L, window)
        kh = _history(k[b], L, capacity, keep)
        vh = _history(v[b], L, capacity, keep)
        for h in range(NH):
            kvh = h // G
            s = (kh[kvh] @ q[b, h].to(torch.float64)) * scale
            s = torch.where(keep, s, torch.tensor(float("-inf"), dtype=torch.float64))
            p = torch.softmax(s, dim=0)
            out[b, h] = p @ vh[kvh]
    return out


def sdpa(q, k, v, lens, B, NH, NKV, HS, capacity, window, scale) -> torch.Tensor:
    """The same through torch.nn.functional.scaled_dot_product_attention."""
    G = NH // NKV
    out = torch.zeros(B, NH, HS, dtype=torch.float64)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        keep = _mask(L, window)
        kh = _history(k[b], L, capacity, keep).repeat_interleave(G, dim=0)  # [NH, L, HS]
        vh = _history(v[b], L, capacity, keep).repeat_interleave(G, dim=0)
        qq = q[b].to(torch.float64).unsqueeze(1)                             # [NH, 1, HS]
        m = keep.view(1, 1, L)
        o = F.scaled_dot_product_attention(qq, kh, vh, attn_mask=m, scale=scale)
        out[b] = o[:, 0, :]
    return out
