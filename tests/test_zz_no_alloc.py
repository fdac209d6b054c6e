"""fd_decode_attn_noalloc, the entry point that allocates nothing, checked on
the GPU through the C ABI against fd_decode_attn_ex and the FP64 oracle.

Some callers cannot allocate device memory while they run: an op executing
inside a serving framework whose memory pool owns the device, or a decode loop
that cannot let cudaMalloc synchronise the device or fail in the middle of a
step. fd_decode_attn_noalloc serves them by keeping its split partials in a
fixed 32 MiB array compiled into libfd.so. This file checks that:

  * two calls in a row - the second finding the first one's partials still in
    that array - each return exactly what the explicit-workspace entry point
    returns for the same plan (the kernels are deterministic, so bit for bit),
    and one of them is within the parity tolerance of the oracle;
  * shapes that use many counters and few, called large, small, large in one
    process, stay exact (no counter left non-zero between calls);
  * the first call of a fresh process, made on a non-blocking stream, is exact
    (the array's one-time clear is ordered before that call's kernels);
  * a shape too large for the array is refused before anything runs;
  * after fd_release, the library-owned workspace and the array are set up
    again on the next call, and both entry points stay exact.

The file is collected last and depends on no other test: it passes alone in a
fresh process and after the rest of the suite.
"""

import ctypes
import subprocess
import sys
import textwrap
from pathlib import Path

import numpy as np
import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import Workload, make_inputs
import oracle
from harness import BF16_EXTRA, bf16_ulp, oracle_ref

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent

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


def _noalloc(lib, w, q, k, v, lens, stream=None):
    out = torch.full_like(q, float("nan"))
    s = torch.cuda.current_stream() if stream is None else stream
    rc = lib.fd_decode_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lens.data_ptr(),
                                    w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, ctypes.c_float(w.scale),
                                    ctypes.c_void_p(s.cuda_stream))
    assert rc == fd.FD_OK, fd.fd_strerror(rc)
    return out


def _assert_same(got, ref, what):
    assert torch.isfinite(got.float()).all(), f"{what}: non-finite output"
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"{what}: differs from fd_decode_attn_ex"


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
    _assert_same(got1, ref1, f"{w.name} call 1")
    _assert_same(got2, ref2, f"{w.name} call 2")
    assert fd.fd_get_device_error() == 0


def test_noalloc_second_call_within_oracle_tolerance():
    """The second of two calls against the FP64 oracle: the bf16 output
    within 1 bf16 ulp + 1e-3 of the oracle rounded to bf16 (this entry point
    writes no fp32 copy, so that half of the parity bar is checked through
    fd_decode_attn_ex, which the calls above match bit for bit)."""
    w = CASES[2]
    lib = fd.load_library()
    _noalloc(lib, w, *_on_device(w, w.seed))
    q, k, v, lens = make_inputs(w, seed=w.seed + 7)
    dev = torch.device("cuda")
    got = _noalloc(lib, w, q.to(dev), k.to(dev), v.to(dev), lens.to(dev))
    torch.cuda.synchronize()
    ref = oracle_ref(w, q, k, v, lens)
    ref16 = oracle.bf16_bits_to_f64(oracle.bf16_round(ref))
    got16 = oracle.bf16_bits_to_f64(got.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.isfinite(got16).all()
    bad = np.abs(got16 - ref16) > bf16_ulp(ref16) + BF16_EXTRA
    assert not bad.any(), f"{bad.sum()} bf16 outputs beyond 1 ulp + 1e-3 of the oracle"


def test_noalloc_large_small_large_shapes_stay_exact():
    """Many counters (B * NKV = 128), then few (1), then many again: each
    call equals fd_decode_attn_ex, so no counter was left non-zero."""
    big = CASES[2]
    small = CASES[1]
    lib = fd.load_library()
    for i, w in enumerate((big, small, big)):
        x = _on_device(w, w.seed + 100 * i)
        ref = _explicit(w, *x)
        got = _noalloc(lib, w, *x)
        torch.cuda.synchronize()
        _assert_same(got, ref, f"{w.name} call {i}")


def test_noalloc_first_call_of_a_process_on_a_nonblocking_stream():
    """In a fresh process, the very first call (which sets the array up) runs
    on a torch side stream, which is non-blocking with respect to the legacy
    stream; its result must equal fd_decode_attn_ex's."""
    script = textwrap.dedent(f"""
        import ctypes, sys
        sys.path.insert(0, {str(ROOT)!r}); sys.path.insert(0, {str(ROOT / 'tests')!r})
        import torch
        import decode_attention_04_gb300 as fd
        from decode_attention_04_gb300.inputs import Workload, make_inputs
        w = Workload("noalloc_fresh", 16, 32, 8, 128, 2048, 0,
                     lens=(1, 2048, 700, 33, 1500, 2, 999, 2047, 64, 65, 1024, 300, 3, 1800, 512, 17), seed=505)
        lib = fd.load_library()
        dev = torch.device("cuda")
        q, k, v, lens = (t.to(dev) for t in make_inputs(w))
        s = torch.cuda.Stream()
        out = torch.full_like(q, float("nan"))
        s.wait_stream(torch.cuda.current_stream())  # inputs and the NaN fill are on the default stream
        with torch.cuda.stream(s):
            rc = lib.fd_decode_attn_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                            lens.data_ptr(), w.B, w.NH, w.NKV, w.HS, w.capacity, w.window,
                                            ctypes.c_float(w.scale), ctypes.c_void_p(s.cuda_stream))
        assert rc == 0, rc
        s.synchronize()
        plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
        ref = torch.empty_like(q)
        fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, None, q, k, v, ref, lens, w.B, w.NH, w.NKV, w.HS,
                             w.capacity, w.window, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "first call differs"
        print("fresh-process first call ok")
    """)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "fresh-process first call ok" in r.stdout


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


def test_release_re_arms_both_library_owned_paths():
    """fd_release frees the library-owned workspaces and forgets the fixed
    array's set-up (the recovery step after a failed call): the next
    fd_decode_attn and fd_decode_attn_noalloc calls set up again - the array
    is cleared again on the caller's stream - and both return exactly what
    fd_decode_attn_ex returns."""
    w = CASES[0]
    lib = fd.load_library()
    q, k, v, lens = _on_device(w, w.seed + 50)
    ref = _explicit(w, q, k, v, lens)
    for i in range(3):
        got_na = _noalloc(lib, w, q, k, v, lens)
        got_lib = torch.full_like(q, float("nan"))
        fd.fd_decode_attn(q, k, v, got_lib, lens, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
        torch.cuda.synchronize()
        _assert_same(got_na, ref, f"noalloc, pass {i}")
        _assert_same(got_lib, ref, f"library workspace, pass {i}")
        fd.fd_release()
    assert fd.fd_get_device_error() == 0
