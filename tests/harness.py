"""GPU test harness: runs libfd.so through the C ABI with guarded buffers and
compares with the FP64 oracle.

Tolerances (the stated acceptance bar for this op):
  * fp32 output (before the bf16 store) vs oracle: max |err| <= 2e-3;
  * bf16 output vs the oracle rounded to bf16: |err| <= 1 bf16 ulp + 1e-3.
"""

from __future__ import annotations

import numpy as np
import torch

import decode_attention_04_gb300 as fd
import oracle

ATOL_F32 = 2e-3
BF16_EXTRA = 1e-3
GUARD = 4096          # bytes of canary on each side of every output buffer
CANARY = 0xA5


class Guarded:
    """A device buffer with canary bytes before and after the usable region."""

    def __init__(self, nbytes: int, device, fill: int | None = None):
        self.nbytes = nbytes
        self.raw = torch.full((GUARD + max(nbytes, 1) + GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.body = self.raw[GUARD:GUARD + max(nbytes, 1)]
        if fill is not None:
            self.body.fill_(fill)

    def view(self, dtype, shape):
        return self.body[: self.nbytes].view(dtype).view(shape)

    def ptr(self) -> int:
        return self.body.data_ptr()

    def canaries_intact(self) -> bool:
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + max(self.nbytes, 1):]
        return bool((lo == CANARY).all().item() and (hi == CANARY).all().item())


def run(w, q, k, v, lens, splits: int = 0, path: int = fd.FD_PATH_AUTO, max_len: int = 0,
        poison_ws: bool = True, device="cuda", inputs_on_device=False, scale=None, cluster: int = 0,
        fused: int = -1, persistent: int = -1, min_len: int = 0):
    """One fd_decode_attn_ex call. Returns dict with out (bf16, cpu), out32
    (fp32, cpu), plan, deverr, canaries (bool). persistent: -1 the plan's
    rule, 0 one block per split, k > 0 a persistent grid of at most k blocks.
    min_len: the plan's lower bound on the lengths (fd_plan_min_len)."""
    dev = torch.device(device)
    if inputs_on_device:
        qd, kd, vd, ld = q, k, v, lens.to(dev)
    else:
        qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, max_len)
    if splits or path or cluster or fused >= 0:
        fd.fd_plan_override(plan, splits, path, cluster, fused)
    set_persistent(plan, persistent)
    if min_len:
        fd.fd_plan_min_len(plan, min_len)
    n = w.B * w.NH * w.HS
    o16 = Guarded(n * 2, dev, fill=0xFF)         # NaN-filled: unwritten rows show up
    o32 = Guarded(n * 4, dev, fill=0xFF)
    ws = Guarded(plan.workspace_bytes, dev, fill=0xFF if poison_ws else 0)
    if plan.workspace_zero_bytes:  # the split counters must start at zero
        ws.body[: plan.workspace_zero_bytes].zero_()
    fd.fd_get_device_error()  # clear
    fd.fd_decode_attn_ex(plan, ws.ptr() if plan.workspace_bytes else None, plan.workspace_bytes, o32.ptr(),
                         qd, kd, vd, o16.ptr(), ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window,
                         w.scale if scale is None else scale)
    torch.cuda.synchronize()
    err = fd.fd_get_device_error()
    counters_zero = bool((ws.body[: plan.workspace_zero_bytes] == 0).all().item()) if plan.workspace_zero_bytes else True
    return dict(out=o16.view(torch.bfloat16, (w.B, w.NH, w.HS)).cpu(),
                out32=o32.view(torch.float32, (w.B, w.NH, w.HS)).cpu(),
                plan=plan, deverr=err, counters_zero=counters_zero,
                canaries=o16.canaries_intact() and o32.canaries_intact() and ws.canaries_intact())


def set_persistent(plan, persistent: int):
    """-1: leave the plan's choice; 0: one block per split; k > 0: a persistent
    grid, narrowed to k blocks when the plan's grid is larger."""
    if persistent < 0:
        return
    fd.fd_plan_persistent(plan, 1 if persistent else 0)
    if 0 < persistent < plan.persistent:
        plan.persistent = persistent


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits); subnormal floor 2^-133."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(np.maximum(e, -126) - 7), 2.0 ** -133)


def check(res: dict, ref: np.ndarray, rows=None, what: str = ""):
    """Assert the GPU result matches the oracle within the tolerances, on all
    rows or on the (b, h) pairs in `rows`."""
    assert res["canaries"], f"{what}: guard canary overwritten"
    assert res["counters_zero"], f"{what}: split counters not back to zero after the call"
    out32 = res["out32"].double().numpy()
    out16 = res["out"].view(torch.int16).numpy().view(np.uint16)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        out32, out16, ref = out32[idx], out16[idx], ref[idx]
    assert np.isfinite(out32).all(), f"{what}: non-finite fp32 output"
    e32 = np.abs(out32 - ref).max()
    assert e32 <= ATOL_F32, f"{what}: fp32 max abs err {e32:.3e} > {ATOL_F32}"
    ref16 = oracle.bf16_bits_to_f64(oracle.bf16_round(ref))
    got16 = oracle.bf16_bits_to_f64(out16)
    lim = bf16_ulp(ref16) + BF16_EXTRA
    bad = np.abs(got16 - ref16) > lim
    assert not bad.any(), f"{what}: {bad.sum()} bf16 outputs beyond 1 ulp + 1e-3 (max {np.abs(got16 - ref16).max():.3e})"
    return e32


def oracle_ref(w, q, k, v, lens, rows=None):
    want = None
    if rows is not None:
        want = np.zeros(w.B * w.NH, dtype=bool)
        for b, h in rows:
            want[b * w.NH + h] = True
    return oracle.decode(q, k, v, lens, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale, want=want)


def run_fp8(w, q, k8, v8, ks, vs, lens, splits: int = 0, max_len: int = 0, device="cuda",
            inputs_on_device=False, scale=None, cluster: int = 0, fused: int = -1, persistent: int = -1,
            min_len: int = 0):
    """One fd_decode_attn_fp8_ex call over an E4M3 cache (codes k8/v8, scales
    ks/vs); same result dict as run()."""
    dev = torch.device(device)
    if inputs_on_device:
        qd, kd, vd, ksd, vsd, ld = q, k8, v8, ks, vs, lens.to(dev)
    else:
        qd, kd, vd, ksd, vsd, ld = (t.to(dev) for t in (q, k8, v8, ks, vs, lens))
    plan = fd.fd_plan_kv(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, max_len, kv_dtype=fd.FD_KV_E4M3)
    if splits or cluster or fused >= 0:
        fd.fd_plan_override(plan, splits, 0, cluster, fused)
    set_persistent(plan, persistent)
    if min_len:
        fd.fd_plan_min_len(plan, min_len)
    n = w.B * w.NH * w.HS
    o16 = Guarded(n * 2, dev, fill=0xFF)
    o32 = Guarded(n * 4, dev, fill=0xFF)
    ws = Guarded(plan.workspace_bytes, dev, fill=0xFF)
    if plan.workspace_zero_bytes:
        ws.body[: plan.workspace_zero_bytes].zero_()
    fd.fd_get_device_error()
    fd.fd_decode_attn_fp8_ex(plan, ws.ptr() if plan.workspace_bytes else None, plan.workspace_bytes, o32.ptr(),
                             qd, kd, vd, ksd, vsd, o16.ptr(), ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window,
                             w.scale if scale is None else scale)
    torch.cuda.synchronize()
    err = fd.fd_get_device_error()
    counters_zero = bool((ws.body[: plan.workspace_zero_bytes] == 0).all().item()) if plan.workspace_zero_bytes else True
    return dict(out=o16.view(torch.bfloat16, (w.B, w.NH, w.HS)).cpu(),
                out32=o32.view(torch.float32, (w.B, w.NH, w.HS)).cpu(),
                plan=plan, deverr=err, counters_zero=counters_zero,
                canaries=o16.canaries_intact() and o32.canaries_intact() and ws.canaries_intact())


def oracle_ref_fp8(w, q, k8, v8, ks, vs, lens, rows=None):
    want = None
    if rows is not None:
        want = np.zeros(w.B * w.NH, dtype=bool)
        for b, h in rows:
            want[b * w.NH + h] = True
    return oracle.decode_fp8(q, k8, v8, ks.cpu().numpy(), vs.cpu().numpy(), lens, w.B, w.NH, w.NKV, w.HS,
                             w.capacity, w.window, w.scale, want=want)
