"""Pin adequacy: plant a plausible mistake in a copy of the oracle source (on
the CPU), build it, and check that the pins catch it.

Each mutant is the oracle with one edit - a dropped term, a wrong sign or
index, a swapped operand, an off-by-one band. The real oracle passes every
check below (test_oracle_pins.py); every mutant must fail at least one.
"""

import ctypes
import json
import subprocess
from pathlib import Path

import numpy as np
import pytest
import torch

from bruteforce import brute_force
from decode_attention_04_gb300.inputs import Workload, make_inputs

ROOT = Path(__file__).resolve().parent.parent
SRC = ROOT / "oracle" / "fd_oracle.cpp"
GOLDEN = Path(__file__).resolve().parent / "golden" / "closed_form.json"

MUTANTS = {
    "group_map_modulo": ("const int kvh = h / group;\n  const int len = p.lens[b];\n  int64_t lo, hi;\n  live_band(p, len, &lo, &hi);\n  const int64_t n = hi - lo;\n  double* o = out + (static_cast<int64_t>(b) * p.NH + h) * p.HS;\n  for (int d = 0; d < p.HS; ++d) o[d] = 0.0;\n  if (n <= 0) return;\n\n  std::vector<double> kb, vb;\n  gather_band(p, b, kvh, lo, hi, kb, vb);\n\n",
                         "const int kvh = h % p.NKV;\n  const int len = p.lens[b];\n  int64_t lo, hi;\n  live_band(p, len, &lo, &hi);\n  const int64_t n = hi - lo;\n  double* o = out + (static_cast<int64_t>(b) * p.NH + h) * p.HS;\n  for (int d = 0; d < p.HS; ++d) o[d] = 0.0;\n  if (n <= 0) return;\n\n  std::vector<double> kb, vb;\n  gather_band(p, b, kvh, lo, hi, kb, vb);\n\n"),
    "slot_off_by_one": ("const int64_t slot = pos % p.capacity;", "const int64_t slot = (pos + 1) % p.capacity;"),
    "band_start_off_by_one": ("static_cast<int64_t>(len) - keep);", "static_cast<int64_t>(len) - keep + 1);"),
    "band_end_off_by_one": ("*hi = len;", "*hi = len > 0 ? len - 1 : 0;"),
    "no_capacity_clamp": ("int64_t keep = std::min<int64_t>(w, p.capacity);", "int64_t keep = w;"),
    "scale_dropped": ("s[i] = p.scale * dot;", "s[i] = dot;"),
    "no_max_shift": ("w[i] = std::exp(s[i] - m);", "w[i] = std::exp(s[i]);"),
    "sign_flipped": ("w[i] = std::exp(s[i] - m);", "w[i] = std::exp(m - s[i]);"),
    "scores_from_values": ("for (int d = 0; d < p.HS; ++d) dot += q[d] * kb[i * p.HS + d];\n    s[i] = p.scale * dot;",
                           "for (int d = 0; d < p.HS; ++d) dot += q[d] * vb[i * p.HS + d];\n    s[i] = p.scale * dot;"),
    "denominator_dropped": ("for (int d = 0; d < p.HS; ++d) o[d] /= denom;", ""),
    "query_row_of_kv_head": ("const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * p.NH + h) * p.HS;\n  for (int d = 0; d < p.HS; ++d) q[d] = bf16_bits_to_double(qrow[d]);\n\n  std::vector<double> s(",
                             "const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * p.NH + kvh) * p.HS;\n  for (int d = 0; d < p.HS; ++d) q[d] = bf16_bits_to_double(qrow[d]);\n\n  std::vector<double> s("),
    "empty_sequence_not_zero": ("  for (int d = 0; d < p.HS; ++d) o[d] = 0.0;\n  if (n <= 0) return;\n\n  std::vector<double> kb, vb;\n  gather_band(p, b, kvh, lo, hi, kb, vb);\n\n  std::vector<double> q(p.HS);\n  const uint16_t* qrow",
                                "  for (int d = 0; d < p.HS; ++d) o[d] = 1.0;\n  if (n <= 0) return;\n  for (int d = 0; d < p.HS; ++d) o[d] = 0.0;\n\n  std::vector<double> kb, vb;\n  gather_band(p, b, kvh, lo, hi, kb, vb);\n\n  std::vector<double> q(p.HS);\n  const uint16_t* qrow"),
}


def _build_mutant(name: str, tmp: Path):
    old, new = MUTANTS[name]
    src = SRC.read_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mpath = tmp / f"{name}.cpp"
    mpath.write_text(src.replace(old, new))
    so = tmp / f"lib{name}.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(mpath), "-o", str(so)],
                   check=True)
    lib = ctypes.CDLL(str(so))
    lib.fd_oracle_decode.restype = ctypes.c_int
    return lib


def _call(lib, q, k, v, lens, B, NH, NKV, HS, cap, win, scale):
    def bits(t):
        return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    qb, kb, vb = bits(q), bits(k), bits(v)
    ln = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    out = np.zeros((B, NH, HS))
    P = ctypes.c_void_p
    lib.fd_oracle_decode(P(qb.ctypes.data), P(kb.ctypes.data), P(vb.ctypes.data), P(ln.ctypes.data),
                         B, NH, NKV, HS, cap, win, ctypes.c_double(scale if scale > 0 else HS ** -0.5),
                         None, 1, P(out.ctypes.data))
    return out


def _golden_failures(lib) -> int:
    fails = 0
    for c in json.loads(GOLDEN.read_text())["cases"]:
        def t(x):
            a = np.vectorize(lambda e: float("nan") if e == "nan" else float(e), otypes=[float])(np.array(x, dtype=object))
            return torch.tensor(a).to(torch.bfloat16)
        out = _call(lib, t(c["q"]), t(c["k"]), t(c["v"]), c["lens"], c["B"], c["NH"], c["NKV"], c["HS"],
                    c["capacity"], c["window"], c["scale"])
        if not np.allclose(out, np.array(c["expected"], float), rtol=0, atol=1e-12, equal_nan=False):
            fails += 1
    return fails


def _brute_failures(lib) -> int:
    fails = 0
    specs = [(1, 8, 2, 128, 64, 0, (41,)), (1, 4, 2, 256, 16, 16, (77,)), (1, 8, 2, 128, 32, 20, (50,)),
             (2, 16, 1, 64, 40, 0, (40, 0)), (1, 8, 2, 64, 16, 0, (40,))]
    for B, NH, NKV, HS, cap, win, lens in specs:
        w = Workload("m", B, NH, NKV, HS, cap, win, lens=lens, seed=3)
        q, k, v, ln = make_inputs(w)
        out = _call(lib, q, k, v, ln, B, NH, NKV, HS, cap, win, w.scale)
        if win <= 0 and max(lens) > cap:
            # the capacity-clamp reading: equal to window = capacity
            ref = _call(lib, q, k, v, ln, B, NH, NKV, HS, cap, cap, w.scale)
        else:
            ref = brute_force(q, k, v, ln, B, NH, NKV, HS, cap, win, w.scale).numpy()
        if not np.allclose(out, ref, rtol=0, atol=1e-12):
            fails += 1
    return fails


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    lib = _build_mutant(name, tmp_path)
    caught = _golden_failures(lib) + _brute_failures(lib)
    assert caught > 0, f"mutant {name} passed every pin"


def test_unmutated_source_passes_the_same_checks(tmp_path):
    so = tmp_path / "libclean.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(SRC), "-o", str(so)], check=True)
    lib = ctypes.CDLL(str(so))
    assert _golden_failures(lib) == 0
    assert _brute_failures(lib) == 0


# ---------------------------------------------------------------- E4M3 form

FP8_MUTANTS = {
    "e4m3_bias_off_by_one": ("std::ldexp(1.0 + m / 8.0, e - 7)", "std::ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_subnormal_as_normal": ("e == 0 ? std::ldexp(m / 8.0, -6)", "e == 0 ? std::ldexp(1.0 + m / 8.0, -7)"),
    "e4m3_every_top_code_nan": ("if (e == 15 && m == 7) return", "if (e == 15) return"),
    "e4m3_sign_dropped": ("return s ? -mag : mag;", "return mag;"),
    "v_scale_dropped": ("e4m3_to_double(p.v8[row * p.HS + d]) * vs;", "e4m3_to_double(p.v8[row * p.HS + d]);"),
    "v_takes_k_scale": ("e4m3_to_double(p.v8[row * p.HS + d]) * vs;", "e4m3_to_double(p.v8[row * p.HS + d]) * ks;"),
    "scale_ignores_sequence": ("const double ks = p.k_scale[static_cast<int64_t>(b) * p.NKV + kvh];",
                               "const double ks = p.k_scale[kvh];"),
}


def _build(src_text: str, name: str, tmp: Path):
    mpath = tmp / f"{name}.cpp"
    mpath.write_text(src_text)
    so = tmp / f"lib{name}.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(mpath), "-o", str(so)],
                   check=True)
    return ctypes.CDLL(str(so))


def _fp8_failures(lib) -> int:
    """The E4M3 pins, restated against torch: the 256-code table equals
    torch's float8_e4m3fn conversion, and the E4M3 form equals float64 SDPA
    over the cache dequantised by torch (per-(sequence, KV head) scales)."""
    from decode_attention_04_gb300.inputs import make_inputs_fp8
    fails = 0
    table = np.zeros(256)
    lib.fd_oracle_e4m3_table(ctypes.c_void_p(table.ctypes.data))
    ref_table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if not (np.array_equal(np.isnan(table), np.isnan(ref_table)) and
            np.array_equal(table[~np.isnan(ref_table)], ref_table[~np.isnan(ref_table)])):
        fails += 1
    for B, NH, NKV, HS, cap, win, lens in [(2, 8, 2, 64, 48, 0, (40, 23)), (2, 16, 1, 128, 32, 20, (70, 5))]:
        w = Workload("m8", B, NH, NKV, HS, cap, win, lens=lens, seed=5)
        q, k8, v8, ks, vs, ln = make_inputs_fp8(w)
        out = np.zeros((B, NH, HS))
        P = ctypes.c_void_p

        def arr(t, dt):
            return np.ascontiguousarray(t.contiguous().numpy().astype(dt, copy=False))
        qb = np.ascontiguousarray(q.contiguous().view(torch.int16).numpy().view(np.uint16))
        kc, vc = arr(k8, np.uint8), arr(v8, np.uint8)
        ksa, vsa = arr(ks, np.float32), arr(vs, np.float32)
        lna = np.ascontiguousarray(np.asarray(ln, dtype=np.int32))
        lib.fd_oracle_decode_fp8(P(qb.ctypes.data), P(kc.ctypes.data), P(vc.ctypes.data), P(ksa.ctypes.data),
                                 P(vsa.ctypes.data), P(lna.ctypes.data), B, NH, NKV, HS, cap, win,
                                 ctypes.c_double(w.scale), None, 1, P(out.ctypes.data))
        kd = k8.view(torch.float8_e4m3fn).to(torch.float64) * ks.double()[:, :, None, None]
        vd = v8.view(torch.float8_e4m3fn).to(torch.float64) * vs.double()[:, :, None, None]
        G = NH // NKV
        keep = min(win if win > 0 else cap, cap)
        for b in range(B):
            L = int(ln[b])
            pos = torch.arange(max(0, L - keep), L)
            kk = kd[b][:, pos % cap].repeat_interleave(G, dim=0)
            vv = vd[b][:, pos % cap].repeat_interleave(G, dim=0)
            o = torch.nn.functional.scaled_dot_product_attention(q[b].double().unsqueeze(1), kk, vv, scale=w.scale)
            if not np.allclose(out[b], o[:, 0].numpy(), rtol=0, atol=1e-12):
                fails += 1
    return fails


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_fp8_pins_catch_planted_mistake(name, tmp_path):
    old, new = FP8_MUTANTS[name]
    src = SRC.read_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    assert _fp8_failures(_build(src.replace(old, new), name, tmp_path)) > 0, f"mutant {name} passed every E4M3 pin"


def test_unmutated_source_passes_the_e4m3_checks(tmp_path):
    assert _fp8_failures(_build(SRC.read_text(), "clean8", tmp_path)) == 0
