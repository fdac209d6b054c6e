"""FP64 CPU oracle for single-token split-KV decode attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library never
imports, links or calls it, and this package imports nothing from the library.

``fd_oracle.cpp`` holds the arithmetic (plain FP64 softmax attention over the
gathered live band, following "Hand-Writing Gemma 4 Flash-Decoding + an FP4
Matvec Bonus (Part 2)", sections "One KV head breaks the textbook" and "The test
that catches what parity misses"). This module only compiles it with g++ and
marshals numpy arrays into it.

Pinning: the attention entry points are pinned by ``tests/test_oracle_pins.py``
(brute force, a library routine, closed forms and invariants); the bf16
helpers ``bf16_round`` and ``bf16_bits_to_f64`` by ``tests/test_oracle_bf16.py``
(torch's conversions where they round once, an exact rational
round-to-nearest-even, every bit pattern, planted mistakes). No function is
"parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "fd_oracle.cpp"
_LIB = _HERE / "libfd_oracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile fd_oracle.cpp into oracle/libfd_oracle.so (portable flags only)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
               str(_SRC), "-o", str(tmp)]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        ci = ctypes.c_int
        lib.fd_oracle_decode.argtypes = [u16p, u16p, u16p, i32p, ci, ci, ci, ci, ci, ci,
                                         ctypes.c_double, u8p, ci, f64p]
        lib.fd_oracle_decode.restype = ci
        lib.fd_oracle_decode_split.argtypes = [u16p, u16p, u16p, i32p, ci, ci, ci, ci, ci, ci,
                                               ctypes.c_double, ci, ci, f64p]
        lib.fd_oracle_decode_split.restype = ci
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.fd_oracle_decode_fp8.argtypes = [u16p, u8p, u8p, f32p, f32p, i32p, ci, ci, ci, ci, ci, ci,
                                             ctypes.c_double, u8p, ci, f64p]
        lib.fd_oracle_decode_fp8.restype = ci
        lib.fd_oracle_e4m3_table.argtypes = [f64p]
        lib.fd_oracle_e4m3_table.restype = None
        _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bit patterns."""
    if not isinstance(a, np.ndarray):
        import torch  # local: numpy callers need no torch
        assert a.dtype == torch.bfloat16, a.dtype
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    assert a.dtype == np.uint16
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_scale(HS: int, scale: float) -> float:
    """scale <= 0 selects 1/sqrt(HS) (the convention of SharpInference issue #156,
    "Background": attnScale <= 0 means 1/sqrt(headDim))."""
    return float(scale) if scale > 0 else 1.0 / float(np.sqrt(HS))


def decode(q, k_cache, v_cache, lens, B, NH, NKV, HS, capacity, window, scale,
           want=None, nthreads: int = 0) -> np.ndarray:
    """FP64 attention output [B, NH, HS] for bf16 inputs q [B,NH,HS] and
    k_cache/v_cache [B,NKV,capacity,HS]; lens int32 [B]; window <= 0 = none.
    ``want`` (bool [B*NH]) restricts the rows computed; the others stay 0."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    assert qb.size == B * NH * HS and kb.size == B * NKV * capacity * HS and vb.size == kb.size
    ln = np.ascontiguousarray(np.asarray(lens, dtype=np.int32).reshape(-1))
    assert ln.size == B
    out = np.zeros((B, NH, HS), dtype=np.float64)
    w = None
    if want is not None:
        w = np.ascontiguousarray(np.asarray(want, dtype=np.uint8).reshape(-1))
        assert w.size == B * NH
    rc = lib.fd_oracle_decode(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                              _ptr(vb, ctypes.c_uint16), _ptr(ln, ctypes.c_int32),
                              B, NH, NKV, HS, capacity, window,
                              default_scale(HS, scale),
                              None if w is None else _ptr(w, ctypes.c_uint8),
                              nthreads, _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("fd_oracle_decode: invalid arguments")
    return out


def decode_split(q, k_cache, v_cache, lens, B, NH, NKV, HS, capacity, window, scale,
                 splits: int, nthreads: int = 0) -> np.ndarray:
    """FP64 split-and-merge restatement (``splits`` contiguous pieces per band)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    ln = np.ascontiguousarray(np.asarray(lens, dtype=np.int32).reshape(-1))
    out = np.zeros((B, NH, HS), dtype=np.float64)
    rc = lib.fd_oracle_decode_split(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                    _ptr(vb, ctypes.c_uint16), _ptr(ln, ctypes.c_int32),
                                    B, NH, NKV, HS, capacity, window,
                                    default_scale(HS, scale), splits, nthreads,
                                    _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("fd_oracle_decode_split: invalid arguments")
    return out


def _codes(a) -> np.ndarray:
    """Accept a torch float8_e4m3fn / uint8 tensor or a uint8 numpy array of E4M3 codes."""
    if not isinstance(a, np.ndarray):
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        a = t.numpy()
    assert a.dtype == np.uint8
    return np.ascontiguousarray(a)


def decode_fp8(q, k8, v8, k_scale, v_scale, lens, B, NH, NKV, HS, capacity, window, scale,
               want=None, nthreads: int = 0) -> np.ndarray:
    """FP64 attention output [B, NH, HS] for bf16 q and an E4M3 cache:
    k8/v8 codes [B,NKV,capacity,HS], k_scale/v_scale fp32 [B,NKV] (value of a
    code = its E4M3 number x the scale of its (sequence, KV head))."""
    lib = _load()
    qb, kc, vc = _bits(q), _codes(k8), _codes(v8)
    assert qb.size == B * NH * HS and kc.size == B * NKV * capacity * HS and vc.size == kc.size
    ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32).reshape(-1))
    vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float32).reshape(-1))
    assert ks.size == B * NKV and vs.size == B * NKV
    ln = np.ascontiguousarray(np.asarray(lens, dtype=np.int32).reshape(-1))
    out = np.zeros((B, NH, HS), dtype=np.float64)
    w = None
    if want is not None:
        w = np.ascontiguousarray(np.asarray(want, dtype=np.uint8).reshape(-1))
    rc = lib.fd_oracle_decode_fp8(_ptr(qb, ctypes.c_uint16), _ptr(kc, ctypes.c_uint8), _ptr(vc, ctypes.c_uint8),
                                  _ptr(ks, ctypes.c_float), _ptr(vs, ctypes.c_float), _ptr(ln, ctypes.c_int32),
                                  B, NH, NKV, HS, capacity, window, default_scale(HS, scale),
                                  None if w is None else _ptr(w, ctypes.c_uint8), nthreads,
                                  _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("fd_oracle_decode_fp8: invalid arguments")
    return out


def e4m3_table() -> np.ndarray:
    """The oracle's value for each of the 256 E4M3 codes."""
    out = np.zeros(256, dtype=np.float64)
    _load().fd_oracle_e4m3_table(_ptr(out, ctypes.c_double))
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even mantissa) and
    return the bit patterns as uint16. The rounding is taken directly from the
    float64 value: the three bf16 neighbours of the float32 image of x bracket
    x, and the nearest of them in float64 wins. NaN maps to 0x7FC0; values
    beyond the largest finite bf16 round to +-inf."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        f = x.astype(np.float32)
    u = f.view(np.uint32).astype(np.int64) & 0xFFFF0000
    sign = u & 0x80000000
    mag = u & 0x7FFF0000
    cands = []
    for step in (-0x10000, 0, 0x10000):
        m = np.clip(mag + step, 0, 0x7F800000)
        cands.append((sign | m).astype(np.uint32))
    vals = [c.view(np.float32).astype(np.float64) for c in cands]
    with np.errstate(invalid="ignore"):
        errs = np.stack([np.abs(v - x) for v in vals])
    best = np.argmin(np.where(np.isnan(errs), np.inf, errs), axis=0)
    bits = np.choose(best, cands)
    # ties: prefer the candidate whose bf16 mantissa LSB is zero
    for i in range(3):
        for j in range(3):
            if i == j:
                continue
            tie = (errs[i] == errs[j]) & (best == i) & (((cands[i] >> 16) & 1) == 1) \
                & (((cands[j] >> 16) & 1) == 0)
            bits = np.where(tie, cands[j], bits)
    r = (bits >> 16).astype(np.uint16)
    # |x| at or above the midpoint between the largest finite bf16,
    # (2 - 2^-7) * 2^127, and 2^128 rounds to infinity (that midpoint is a tie
    # whose even neighbour is the infinity encoding).
    over = np.abs(x) >= (2.0 - 2.0 ** -8) * 2.0 ** 127
    r = np.where(over, np.where(x > 0, 0x7F80, 0xFF80).astype(np.uint16), r)
    r = np.where(np.isnan(x), np.uint16(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


__all__ = ["build", "decode", "decode_split", "decode_fp8", "e4m3_table", "default_scale", "bf16_round",
           "bf16_bits_to_f64"]
