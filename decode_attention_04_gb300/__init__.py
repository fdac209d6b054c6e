"""Python binding of libfd.so: single-token split-KV decode attention
(Flash-Decoding) over a position-addressed bf16 or FP8 (E4M3) KV cache on GB300.

Every function here has the name of the C entry point it wraps
(include/fd_decode_attn.h) and only marshals arguments: torch tensors become
device pointers, the current torch stream becomes the CUDA stream, non-zero
status codes become FdError. All arithmetic runs in libfd.so's kernels. There
is no fallback: if libfd.so is missing or a call fails, an exception is raised.
Where Python headers were available at build time, fd_decode_attn and
fd_decode_attn_fp8 go through the small compiled module _fdfast (the same
libfd.so, less host time per call); elsewhere they go through ctypes.

Typical use in a decode loop (every layer its own cache; lens counts the
current token, whose K/V are already in the cache):

    import torch, decode_attention_04_gb300 as fd
    # q: bf16 [B, NH, HS]; k, v: bf16 [B, NKV, capacity, HS]; lens: int32 [B]
    out = fd.decode_attention(q, k, v, lens, window=1024)      # allocates out
    fd.fd_decode_attn(q, k, v, out, lens, B, NH, NKV, HS, capacity, window,
                      0.0)                                      # into out

The first call for a (device, stream) sizes the library's workspace; later
calls may be captured in a CUDA graph. fd_plan / fd_decode_attn_ex take an
explicit plan and workspace instead (nothing allocated by the library), and
fd_decode_attn_noalloc uses a fixed scratch array compiled into libfd.so.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libfd.so"

FD_OK = 0
FD_ERR_INVALID_ARG = 1
FD_ERR_UNSUPPORTED = 2
FD_ERR_ALIGNMENT = 3
FD_ERR_CUDA = 4
FD_ERR_WORKSPACE = 5
FD_ERR_SCRATCH_LIMIT = 6
FD_NOALLOC_SCRATCH_BYTES = 32 << 20

FD_DEVERR_LEN_NEGATIVE = 1 << 0
FD_DEVERR_LEN_CLAMPED = 1 << 1
FD_DEVERR_WAIT_TIMEOUT = 1 << 2
FD_DEVERR_MIN_LEN = 1 << 3

FD_PATH_AUTO = 0
FD_PATH_SIMT = 1
FD_PATH_TC = 2
FD_PATH_UMMA = 3

FD_KV_BF16 = 0
FD_KV_E4M3 = 1

EXPORTED = ["fd_plan", "fd_plan_sms", "fd_plan_kv", "fd_plan_sms_kv", "fd_plan_override", "fd_plan_persistent",
            "fd_plan_min_len", "fd_workspace_bytes",
            "fd_decode_attn", "fd_decode_attn_ex", "fd_decode_attn_fp8", "fd_decode_attn_fp8_ex",
            "fd_decode_attn_noalloc", "fd_debug_withhold_copies", "fd_get_device_error", "fd_release",
            "fd_strerror", "fd_version"]


class fd_plan_t(ctypes.Structure):
    _fields_ = [
        ("num_splits", ctypes.c_int),
        ("path", ctypes.c_int),
        ("cluster", ctypes.c_int),
        ("granule", ctypes.c_int),
        ("max_band", ctypes.c_int),
        ("ctas_per_sm", ctypes.c_int),
        ("num_sms", ctypes.c_int),
        ("max_cluster", ctypes.c_int),
        ("fused", ctypes.c_int),
        ("group_bytes", ctypes.c_int),
        ("kv_dtype", ctypes.c_int),
        ("consumer_warps", ctypes.c_int),
        ("persistent", ctypes.c_int),
        ("min_len", ctypes.c_int),
        ("workspace_bytes", ctypes.c_size_t),
        ("workspace_zero_bytes", ctypes.c_size_t),
        ("B", ctypes.c_int),
        ("NH", ctypes.c_int),
        ("NKV", ctypes.c_int),
        ("HS", ctypes.c_int),
        ("capacity", ctypes.c_int),
        ("window", ctypes.c_int),
    ]

    def __repr__(self):
        return "fd_plan_t(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class FdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fd_strerror(status)} (status {status})")


_lib = None


def load_library(path: Path | str | None = None):
    """Load libfd.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(python -m decode_attention_04_gb300.build)")
    lib = ctypes.CDLL(str(p))
    ci, vp, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    planp = ctypes.POINTER(fd_plan_t)
    sig = {
        "fd_plan": (ci, [ci, ci, ci, ci, ci, ci, ci, ci, planp]),
        "fd_plan_sms": (ci, [ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, planp]),
        "fd_plan_kv": (ci, [ci, ci, ci, ci, ci, ci, ci, ci, ci, planp]),
        "fd_plan_sms_kv": (ci, [ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, planp]),
        "fd_plan_override": (ci, [planp, ci, ci, ci, ci]),
        "fd_plan_persistent": (ci, [planp, ci]),
        "fd_plan_min_len": (ci, [planp, ci]),
        "fd_debug_withhold_copies": (ci, [ci, ctypes.c_ulonglong]),
        "fd_workspace_bytes": (sz, [planp]),
        "fd_decode_attn": (ci, [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, vp]),
        "fd_decode_attn_ex": (ci, [planp, vp, sz, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci,
                                   ctypes.c_float, vp]),
        "fd_decode_attn_fp8": (ci, [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, vp]),
        "fd_decode_attn_fp8_ex": (ci, [planp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci,
                                       ctypes.c_float, vp]),
        "fd_decode_attn_noalloc": (ci, [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ctypes.c_float, vp]),
        "fd_get_device_error": (ci, [vp, ctypes.POINTER(ctypes.c_uint)]),
        "fd_release": (None, []),
        "fd_strerror": (ctypes.c_char_p, [ci]),
        "fd_version": (ci, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != FD_OK:
        raise FdError(rc, where)


def fd_strerror(status: int) -> str:
    return load_library().fd_strerror(status).decode()


def fd_version() -> int:
    return load_library().fd_version()


def fd_plan(B, NH, NKV, HS, capacity, window, max_len=0, device=None) -> fd_plan_t:
    if device is None:
        import torch
        device = torch.cuda.current_device()
    p = fd_plan_t()
    _check(load_library().fd_plan(B, NH, NKV, HS, capacity, window, max_len, int(device), ctypes.byref(p)),
           "fd_plan")
    return p


def fd_plan_sms(B, NH, NKV, HS, capacity, window, max_len, num_sms, ctas_per_sm, max_cluster=8) -> fd_plan_t:
    p = fd_plan_t()
    _check(load_library().fd_plan_sms(B, NH, NKV, HS, capacity, window, max_len, num_sms, ctas_per_sm,
                                      max_cluster, ctypes.byref(p)), "fd_plan_sms")
    return p


def fd_plan_kv(B, NH, NKV, HS, capacity, window, max_len=0, device=None, kv_dtype=FD_KV_BF16) -> fd_plan_t:
    if device is None:
        import torch
        device = torch.cuda.current_device()
    p = fd_plan_t()
    _check(load_library().fd_plan_kv(B, NH, NKV, HS, capacity, window, max_len, int(device), int(kv_dtype),
                                     ctypes.byref(p)), "fd_plan_kv")
    return p


def fd_plan_sms_kv(B, NH, NKV, HS, capacity, window, max_len, num_sms, ctas_per_sm, max_cluster=8,
                   kv_dtype=FD_KV_BF16) -> fd_plan_t:
    p = fd_plan_t()
    _check(load_library().fd_plan_sms_kv(B, NH, NKV, HS, capacity, window, max_len, num_sms, ctas_per_sm,
                                         max_cluster, int(kv_dtype), ctypes.byref(p)), "fd_plan_sms_kv")
    return p


def fd_plan_override(plan: fd_plan_t, num_splits: int = 0, path: int = FD_PATH_AUTO, cluster: int = 0,
                     fused: int = -1) -> fd_plan_t:
    _check(load_library().fd_plan_override(ctypes.byref(plan), num_splits, path, cluster, fused),
           "fd_plan_override")
    return plan


def fd_plan_persistent(plan: fd_plan_t, persistent: int = 1) -> fd_plan_t:
    _check(load_library().fd_plan_persistent(ctypes.byref(plan), persistent), "fd_plan_persistent")
    return plan


def fd_plan_min_len(plan: fd_plan_t, min_len: int) -> fd_plan_t:
    """Record the caller's lower bound on every len_b (tiles of slots that any
    such length makes live may then be read before the lengths arrive)."""
    _check(load_library().fd_plan_min_len(ctypes.byref(plan), int(min_len)), "fd_plan_min_len")
    return plan


def fd_debug_withhold_copies(withhold_tile: int, wait_limit_ns: int = 0) -> None:
    """Test hook of the bounded waits: split blocks issue no copies from
    their tile `withhold_tile` on (< 0: off), and waits give up after
    `wait_limit_ns` (0: the default, about one second)."""
    _check(load_library().fd_debug_withhold_copies(int(withhold_tile), int(wait_limit_ns)),
           "fd_debug_withhold_copies")


def fd_workspace_bytes(plan: fd_plan_t) -> int:
    return load_library().fd_workspace_bytes(ctypes.byref(plan))


_fast_mod = None
_fast_for = None  # the ctypes handle the compiled entries belong to


def _fast():
    """The compiled CPython entries (``_fdfast``, linked to the in-tree
    libfd.so) when they were built and that library is the one loaded; else
    None, and calls go through ctypes."""
    global _fast_mod, _fast_for
    lib = load_library()
    if _fast_for is not lib:
        _fast_for, _fast_mod = lib, None
        if Path(getattr(lib, "_name", "")).resolve() == LIB_PATH.resolve():
            try:
                from . import _fdfast
                _fast_mod = _fdfast
            except ImportError:
                _fast_mod = None
    return _fast_mod


def fd_decode_attn(q, k_cache, v_cache, out, lens, B, NH, NKV, HS, capacity, window, scale,
                   stream=None) -> None:
    f = _fast()
    if f is not None:
        rc = f.decode_attn(_ptr(q) or 0, _ptr(k_cache) or 0, _ptr(v_cache) or 0, _ptr(out) or 0, _ptr(lens) or 0,
                           B, NH, NKV, HS, capacity, window, float(scale), _stream(stream) or 0)
    else:
        rc = load_library().fd_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lens),
                                           B, NH, NKV, HS, capacity, window, float(scale), _stream(stream))
    _check(rc, "fd_decode_attn")


def fd_decode_attn_ex(plan: fd_plan_t, workspace, workspace_bytes, out_f32, q, k_cache, v_cache, out, lens,
                      B, NH, NKV, HS, capacity, window, scale, stream=None) -> None:
    f = _fast()
    if f is not None:
        rc = f.decode_attn_ex(ctypes.addressof(plan), _ptr(workspace) or 0, int(workspace_bytes), _ptr(out_f32) or 0,
                              _ptr(q) or 0, _ptr(k_cache) or 0, _ptr(v_cache) or 0, _ptr(out) or 0, _ptr(lens) or 0,
                              B, NH, NKV, HS, capacity, window, float(scale), _stream(stream) or 0)
    else:
        rc = load_library().fd_decode_attn_ex(ctypes.byref(plan), _ptr(workspace), int(workspace_bytes),
                                              _ptr(out_f32), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                              _ptr(lens), B, NH, NKV, HS, capacity, window, float(scale),
                                              _stream(stream))
    _check(rc, "fd_decode_attn_ex")


def fd_decode_attn_fp8(q, k8, v8, k_scale, v_scale, out, lens, B, NH, NKV, HS, capacity, window, scale,
                       stream=None) -> None:
    f = _fast()
    if f is not None:
        rc = f.decode_attn_fp8(_ptr(q) or 0, _ptr(k8) or 0, _ptr(v8) or 0, _ptr(k_scale) or 0, _ptr(v_scale) or 0,
                               _ptr(out) or 0, _ptr(lens) or 0, B, NH, NKV, HS, capacity, window, float(scale),
                               _stream(stream) or 0)
    else:
        rc = load_library().fd_decode_attn_fp8(_ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale), _ptr(out),
                                               _ptr(lens), B, NH, NKV, HS, capacity, window, float(scale),
                                               _stream(stream))
    _check(rc, "fd_decode_attn_fp8")


def fd_decode_attn_fp8_ex(plan: fd_plan_t, workspace, workspace_bytes, out_f32, q, k8, v8, k_scale, v_scale, out,
                          lens, B, NH, NKV, HS, capacity, window, scale, stream=None) -> None:
    f = _fast()
    if f is not None:
        rc = f.decode_attn_fp8_ex(ctypes.addressof(plan), _ptr(workspace) or 0, int(workspace_bytes),
                                  _ptr(out_f32) or 0, _ptr(q) or 0, _ptr(k8) or 0, _ptr(v8) or 0, _ptr(k_scale) or 0,
                                  _ptr(v_scale) or 0, _ptr(out) or 0, _ptr(lens) or 0, B, NH, NKV, HS, capacity,
                                  window, float(scale), _stream(stream) or 0)
    else:
        rc = load_library().fd_decode_attn_fp8_ex(ctypes.byref(plan), _ptr(workspace), int(workspace_bytes),
                                                  _ptr(out_f32), _ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale),
                                                  _ptr(v_scale), _ptr(out), _ptr(lens), B, NH, NKV, HS, capacity,
                                                  window, float(scale), _stream(stream))
    _check(rc, "fd_decode_attn_fp8_ex")


def fd_decode_attn_noalloc(q, k_cache, v_cache, out, lens, B, NH, NKV, HS, capacity, window, scale,
                           stream=None) -> None:
    """fd_decode_attn for callers that must not allocate device memory while
    they run: the split partials go to a fixed 32 MiB array inside libfd.so.
    Calls that overlap on the GPU share that array and race; serialise them."""
    _check(load_library().fd_decode_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lens),
                                                 B, NH, NKV, HS, capacity, window, float(scale),
                                                 _stream(stream)),
           "fd_decode_attn_noalloc")


def fd_get_device_error(stream=None) -> int:
    err = ctypes.c_uint(0)
    _check(load_library().fd_get_device_error(_stream(stream), ctypes.byref(err)), "fd_get_device_error")
    return err.value


def fd_release() -> None:
    load_library().fd_release()


def decode_attention(q, k_cache, v_cache, lens, window=0, scale=0.0, out=None, stream=None):
    """Convenience form over torch tensors: q [B,NH,HS], caches [B,NKV,capacity,HS]
    (bf16, CUDA), lens int32 [B] (CUDA). Allocates `out` if not given and calls
    fd_decode_attn."""
    import torch
    B, NH, HS = q.shape
    _, NKV, capacity, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    fd_decode_attn(q, k_cache, v_cache, out, lens, B, NH, NKV, HS, capacity, window, scale, stream)
    return out


__all__ = EXPORTED + ["fd_plan_t", "FdError", "load_library", "decode_attention", "LIB_PATH"]
