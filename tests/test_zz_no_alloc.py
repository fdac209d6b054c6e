"""fd_decode_attn_noalloc, the entry point that allocates nothing, checked on
the GPU through the C ABI against fd_decode_attn_ex.

Some callers cannot allocate device memory while they run: an op executing
inside a serving framework whose memory pool owns the device, or a decode loop
that cannot let cudaMalloc synchronise the device or fail in the middle of a
step. fd_decode_attn_noalloc serves them by keeping its split partials in a
fixed 32 MiB array compiled into libfd.so. This file checks that two calls in
a row - the second one finding the first one's partials still in that array -
each return what the explicit-workspace entry point returns, within the bf16
tolerance the parity tests use, and that a shape too large for the array is
refused before anything runs.

The file is collected last and depends on no other test: it passes alone in a
fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import Workload, make_inputs
from harness import BF16_EXTRA, bf16_ulp

pytestmark = pytest.mark.gpu

CASES = [
    Workload("noalloc_ring", 1, 16, 8, 256, 1024, 1024, lens=(5000,), seed=501),
    Workload("noalloc_mqa", 2, 16, 1, 512, 4096, 0, lens=(4096, 1234), seed=502),
    Workload("noalloc_ragged", 16, 32, 8, 128, 2048, 0,
             lens=(1, 2048, 700, 33, 1500, 2, 999, 2047, 64, 65, 1024, 300, 3, 1800, 512, 17), seed=503),
]


def _on_device(w, seed):
    q, k, v, lens = make_inputs(w, seed=seed)
    dev = torch.device("cuda")
    return q.to(dev), k.to(dev), v.to(dev), lens.to(dev)


def _explicit(w, q, k, v, lens):
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    ws = torch.zeros(max(1, plan.workspace_bytes), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, None, q, k, v, out, lens, w.B, w.NH, w.NKV, w.HS,
                         w.capacity, w.window, w.scale)
    return out


def _noalloc(lib, w, q, k, v, lens):
    out = torch.full_like(q, float("nan"))
    rc = lib.fd_decode_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lens.data_ptr(),
                                    w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, ctypes.c_float(w.scale),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fd.FD_OK, fd.fd_strerror(rc)
    return out


def _assert_close(got, ref, what):
    x = got.double().cpu().numpy()
    y = ref.double().cpu().numpy()
    assert np.isfinite(x).all(), f"{what}: non-finite output"
    bad = np.abs(x - y) > bf16_ulp(y) + BF16_EXTRA
    assert not bad.any(), f"{what}: {bad.sum()} outputs beyond 1 bf16 ulp + 1e-3"


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_explicit_workspace_on_two_calls_in_a_row(w):
    lib = fd.load_library()
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    assert 0 < plan.workspace_bytes <= fd.FD_NOALLOC_SCRATCH_BYTES
    first = _on_device(w, w.seed)
    second = _on_device(w, w.seed + 1000)
    ref1 = _explicit(w, *first)
    ref2 = _explicit(w, *second)
    got1 = _noalloc(lib, w, *first)
    got2 = _noalloc(lib, w, *second)
    torch.cuda.synchronize()
    _assert_close(got1, ref1, f"{w.name} call 1")
    _assert_close(got2, ref2, f"{w.name} call 2")
    assert fd.fd_get_device_error() == 0


def test_noalloc_refuses_a_shape_beyond_its_scratch():
    lib = fd.load_library()
    # 16 sequences of the 131072-position MQA geometry: the plan's split
    # partials need more than the fixed array holds.
    B, NH, NKV, HS, cap = 16, 16, 1, 512, 131072
    plan = fd.fd_plan(B, NH, NKV, HS, cap, 0)
    assert plan.workspace_bytes > fd.FD_NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda")
    # Real buffers of the full size, so nothing could read out of bounds even
    # if the refusal were missing; lens are tiny.
    q = torch.zeros(B, NH, HS, dtype=torch.bfloat16, device=dev)
    k = torch.empty(B, NKV, cap, HS, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    lens = torch.ones(B, dtype=torch.int32, device=dev)
    out = torch.full_like(q, 7.0)
    rc = lib.fd_decode_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lens.data_ptr(),
                                    B, NH, NKV, HS, cap, 0, ctypes.c_float(0.0),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fd.FD_ERR_SCRATCH_LIMIT
    assert "32 MiB" in fd.fd_strerror(rc)
    torch.cuda.synchronize()
    assert (out == 7.0).all()
