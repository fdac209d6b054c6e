"""Pins for the FP64 oracle (CPU only).

The oracle is pinned to things other than itself:
  * hand-derived closed forms (tests/golden/closed_form.json);
  * a naive full-history masked-softmax brute force and torch's
    scaled_dot_product_attention in float64 (library routine), on tiny inputs
    of every geometry, scaled down;
  * invariants the page states or implies ("Hand-Writing Gemma 4
    Flash-Decoding + an FP4 Matvec Bonus (Part 2)", sections "One KV head
    breaks the textbook" and "The test that catches what parity misses"):
    window >= len equals no window, ring wrap equals the contiguously
    reordered cache, split count does not change the result, a one-position
    band returns V exactly, NaN outside the band never reaches the output;
  * closed forms: K = 0 gives the band mean of V, constant V gives V, one
    dominant key gives its V, permuting (K, V) pairs in the band changes nothing.
"""

import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

from bruteforce import brute_force, sdpa
from decode_attention_04_gb300.inputs import Workload, live_slots, make_inputs

GOLDEN = Path(__file__).resolve().parent / "golden" / "closed_form.json"


def _bf16(nested) -> torch.Tensor:
    arr = np.array(nested, dtype=object)
    f = np.vectorize(lambda x: float("nan") if x == "nan" else float(x), otypes=[np.float64])(arr)
    t = torch.tensor(f, dtype=torch.float64).to(torch.bfloat16)
    # exactness of the fixture: every finite value must be a bf16 value
    back = t.to(torch.float64).numpy()
    fin = np.isfinite(f)
    assert np.array_equal(back[fin], f[fin]), "fixture value not exact in bf16"
    return t


def _run(oracle_mod, q, k, v, lens, w: dict, **kw):
    return oracle_mod.decode(q, k, v, lens, w["B"], w["NH"], w["NKV"], w["HS"],
                             w["capacity"], w["window"], w["scale"], **kw)


# ---------------------------------------------------------------- closed forms

_CASES = json.loads(GOLDEN.read_text())["cases"]


@pytest.mark.parametrize("case", _CASES, ids=[c["name"] for c in _CASES])
def test_golden_closed_form(case, oracle_mod):
    q, k, v = _bf16(case["q"]), _bf16(case["k"]), _bf16(case["v"])
    lens = torch.tensor(case["lens"], dtype=torch.int32)
    out = _run(oracle_mod, q, k, v, lens, case)
    exp = np.array(case["expected"], dtype=np.float64)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-12)


# -------------------------------------------------------- brute force, library

TINY = [
    # B, NH, NKV, HS, capacity, window, lens           (what it scales down)
    (1, 8, 2, 128, 64, 0, (41,)),                       # Llama 8x4 grouping
    (1, 4, 2, 256, 16, 16, (77,)),                      # Gemma local ring, wrapped
    (1, 16, 1, 512, 48, 0, (33,)),                      # Gemma global MQA d512
    (2, 16, 1, 64, 40, 0, (40, 7)),                     # MQA, full cache + short
    (1, 8, 2, 128, 32, 20, (50,)),                      # ring with window < capacity
    (3, 2, 2, 64, 64, 0, (1, 64, 17)),                  # MHA (G = 1), ragged
    (2, 4, 4, 64, 8, 3, (9, 2)),                        # tiny window
    (2, 8, 1, 128, 24, 24, (0, 60)),                    # empty sequence in a batch
]


def _tiny(spec, seed=7, poison=True):
    B, NH, NKV, HS, cap, win, lens = spec
    w = Workload("tiny", B, NH, NKV, HS, cap, win, lens=lens, seed=seed)
    q, k, v, ln = make_inputs(w, poison=poison)
    return w, q, k, v, ln


def _wdict(w):
    return dict(B=w.B, NH=w.NH, NKV=w.NKV, HS=w.HS, capacity=w.capacity, window=w.window, scale=w.scale)


@pytest.mark.parametrize("spec", TINY)
def test_oracle_equals_bruteforce_and_sdpa(spec, oracle_mod):
    w, q, k, v, ln = _tiny(spec)
    o1 = _run(oracle_mod, q, k, v, ln, _wdict(w))
    args = (q, k, v, ln, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    o2 = brute_force(*args).numpy()
    o3 = sdpa(*args).numpy()
    assert np.isfinite(o1).all()
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o1, o3, rtol=0, atol=1e-12)


def test_mha_is_per_head_sdpa(oracle_mod):
    """G = 1 (NKV = NH): every head is plain single-query attention."""
    w, q, k, v, ln = _tiny((2, 4, 4, 64, 32, 0, (32, 19)), seed=11)
    o1 = _run(oracle_mod, q, k, v, ln, _wdict(w))
    for b in range(w.B):
        L = int(ln[b])
        for h in range(w.NH):
            qq = q[b, h].double().view(1, 1, -1)
            kk = k[b, h, :L].double().unsqueeze(0)
            vv = v[b, h, :L].double().unsqueeze(0)
            ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=w.scale)
            np.testing.assert_allclose(o1[b, h], ref.view(-1).numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ invariants

def test_window_at_least_len_equals_no_window(oracle_mod):
    w, q, k, v, ln = _tiny((2, 8, 2, 128, 64, 0, (50, 64)), seed=3)
    base = _run(oracle_mod, q, k, v, ln, _wdict(w))
    for win in (64, 50, 60):
        d = _wdict(w)
        d["window"] = win
        got = _run(oracle_mod, q, k, v, ln, d)
        assert np.array_equal(got[0], base[0])          # len 50 <= window
        if win >= 64:
            assert np.array_equal(got[1], base[1])      # len 64 <= window
        else:
            assert not np.allclose(got[1], base[1])     # window cuts sequence 1


def test_no_window_beyond_capacity_keeps_last_capacity_positions(oracle_mod):
    """Reading: a cache holds at most `capacity` positions, so with no window and
    len > capacity the band is the last `capacity` positions - the same as a
    window equal to the capacity."""
    w, q, k, v, ln = _tiny((1, 8, 2, 128, 32, 32, (81,)), seed=4)
    d = _wdict(w)
    win = _run(oracle_mod, q, k, v, ln, d)
    d["window"] = 0
    assert np.array_equal(_run(oracle_mod, q, k, v, ln, d), win)


def test_ring_wrap_equals_contiguous_reordering(oracle_mod):
    cap, win, L = 16, 16, 53
    w, q, k, v, ln = _tiny((1, 4, 2, 64, cap, win, (L,)), seed=5)
    # contiguous cache of capacity >= len holding position p at slot p
    cap2 = 64
    k2 = torch.full((1, 2, cap2, 64), float("nan")).to(torch.bfloat16)
    v2 = k2.clone()
    for p in range(L - win, L):
        k2[0, :, p] = k[0, :, p % cap]
        v2[0, :, p] = v[0, :, p % cap]
    ring = _run(oracle_mod, q, k, v, ln, _wdict(w))
    d = _wdict(w)
    d.update(capacity=cap2, window=win)
    flat = _run(oracle_mod, q, k2, v2, ln, d)
    assert np.array_equal(ring, flat)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 19, 53, 200])
def test_split_merge_is_exact(splits, oracle_mod):
    w, q, k, v, ln = _tiny((2, 8, 2, 128, 64, 0, (53, 5)), seed=9)
    plain = _run(oracle_mod, q, k, v, ln, _wdict(w))
    split = oracle_mod.decode_split(q, k, v, ln, w.B, w.NH, w.NKV, w.HS, w.capacity,
                                    w.window, w.scale, splits)
    np.testing.assert_allclose(split, plain, rtol=0, atol=1e-12)


def test_single_position_band_returns_v_exactly(oracle_mod):
    # len = 1
    w, q, k, v, ln = _tiny((1, 8, 2, 128, 32, 0, (1,)), seed=13)
    out = _run(oracle_mod, q, k, v, ln, _wdict(w))
    for h in range(8):
        assert np.array_equal(out[0, h], v[0, h // 4, 0].double().numpy())
    # window = 1 on a wrapped ring: the band is position len-1 alone
    w, q, k, v, ln = _tiny((1, 8, 2, 128, 16, 1, (37,)), seed=14)
    out = _run(oracle_mod, q, k, v, ln, _wdict(w))
    for h in range(8):
        assert np.array_equal(out[0, h], v[0, h // 4, 36 % 16].double().numpy())


def _band_positions(L, cap, win):
    """Positions held live after writing tokens 0..L-1 at slot p % cap, by
    simulation: the latest writer of each slot, kept if within the window."""
    owner = {}
    for p in range(L):
        owner[p % cap] = p
    keep = cap if win <= 0 else min(win, cap)
    return sorted(p for p in owner.values() if p >= L - keep)


def test_zero_keys_give_band_mean(oracle_mod):
    cap, win, L = 32, 20, 77
    w, q, k, v, ln = _tiny((1, 8, 2, 128, cap, win, (L,)), seed=15)
    k = torch.where(torch.isnan(k), k, torch.zeros_like(k))  # keep poison, zero the rest
    out = _run(oracle_mod, q, k, v, ln, _wdict(w))
    pos = _band_positions(L, cap, win)
    assert len(pos) == 20
    for h in range(8):
        rows = v[0, h // 4, [p % cap for p in pos]].double().numpy()
        np.testing.assert_allclose(out[0, h], rows.mean(axis=0), rtol=0, atol=1e-12)


def test_constant_values_give_that_value(oracle_mod):
    w, q, k, v, ln = _tiny((2, 16, 1, 512, 40, 0, (40, 23)), seed=16)
    row = torch.randn(512, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    v = torch.where(torch.isnan(v), v, row.view(1, 1, 1, 512).expand_as(v))
    out = _run(oracle_mod, q, k, v, ln, _wdict(w))
    np.testing.assert_allclose(out, np.broadcast_to(row.double().numpy(), out.shape), rtol=0, atol=1e-12)


def test_one_dominant_key_returns_its_value(oracle_mod):
    w, q, k, v, ln = _tiny((1, 4, 1, 64, 64, 0, (50,)), seed=17)
    j = 31
    # k_j = 64 q (power-of-two scaling is exact in bf16): score 64*|q|^2/8 >> others
    k = k.clone()
    k[0, 0, j] = (q[0, 0].double() * 64).to(torch.bfloat16)
    out = _run(oracle_mod, q, k, v, ln, _wdict(w))
    np.testing.assert_allclose(out[0, 0], v[0, 0, j].double().numpy(), rtol=0, atol=1e-12)


def test_permuting_band_pairs_changes_nothing(oracle_mod):
    cap, win, L = 32, 24, 70
    w, q, k, v, ln = _tiny((1, 8, 2, 128, cap, win, (L,)), seed=18)
    slots = [p % cap for p in _band_positions(L, cap, win)]
    perm = np.random.default_rng(0).permutation(len(slots))
    k2, v2 = k.clone(), v.clone()
    for a, bidx in zip(slots, perm):
        k2[0, :, a] = k[0, :, slots[bidx]]
        v2[0, :, a] = v[0, :, slots[bidx]]
    o1 = _run(oracle_mod, q, k, v, ln, _wdict(w))
    o2 = _run(oracle_mod, q, k2, v2, ln, _wdict(w))
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_nan_poison_outside_band_never_reaches_output(oracle_mod):
    for spec in TINY:
        w, q, k, v, ln = _tiny(spec, seed=19)
        out = _run(oracle_mod, q, k, v, ln, _wdict(w))
        assert np.isfinite(out).all(), spec


def test_nan_inside_band_reaches_exactly_its_group(oracle_mod):
    """Harness self-test: a NaN planted in a live slot must surface, and only in
    the Q heads of the KV head it was planted in."""
    cap, win, L = 32, 0, 29
    w, q, k, v, ln = _tiny((1, 8, 2, 128, cap, win, (L,)), seed=20)
    nan = torch.tensor(float("nan")).to(torch.bfloat16)
    for which in ("k", "v"):
        kk, vv = k.clone(), v.clone()
        (kk if which == "k" else vv)[0, 1, 11, 5] = nan
        out = _run(oracle_mod, q, kk, vv, ln, _wdict(w))
        assert np.isfinite(out[0, :4]).all()
        if which == "k":
            assert np.isnan(out[0, 4:]).all()
        else:
            assert np.isnan(out[0, 4:, 5]).all()


def test_live_slots_matches_write_simulation():
    for L, cap, win in [(0, 8, 0), (5, 8, 0), (8, 8, 0), (53, 16, 16), (53, 16, 10), (7, 16, 3), (100, 32, 1)]:
        live = set(p % cap for p in _band_positions(L, cap, win))
        mask = live_slots(L, cap, win)
        assert set(mask.nonzero().view(-1).tolist()) == live


def test_sampled_rows_equal_full(oracle_mod):
    w, q, k, v, ln = _tiny((2, 16, 1, 512, 40, 0, (40, 23)), seed=21)
    full = _run(oracle_mod, q, k, v, ln, _wdict(w))
    want = np.zeros(w.B * w.NH, dtype=bool)
    want[[0, 5, 17, 31]] = True
    part = _run(oracle_mod, q, k, v, ln, _wdict(w), want=want)
    for r in range(w.B * w.NH):
        b, h = divmod(r, w.NH)
        if want[r]:
            assert np.array_equal(part[b, h], full[b, h])
        else:
            assert not part[b, h].any()


# ------------------------------------------------------- FP8 (E4M3) cache form

def test_e4m3_decoding_matches_library_for_every_code(oracle_mod):
    """The oracle's E4M3 values (from the format's definition) equal torch's
    float8_e4m3fn conversion for all 256 codes, NaN codes included."""
    ours = oracle_mod.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ours)
    assert np.array_equal(ours[fin], ref[fin])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9  # largest finite, smallest subnormal


def _fp8_case(spec, seed):
    from decode_attention_04_gb300.inputs import make_inputs_fp8
    B, NH, NKV, HS, cap, win, lens = spec
    w = Workload("tiny8", B, NH, NKV, HS, cap, win, lens=lens, seed=seed)
    return (w, *make_inputs_fp8(w))


@pytest.mark.parametrize("spec", TINY[:6])
def test_fp8_form_equals_bf16_form_on_exact_values(spec, oracle_mod):
    """With power-of-two scales every dequantised value is a bf16 value; the
    FP8 form must then give exactly the bf16 oracle's result."""
    w, q, k8, v8, ks, vs, ln = _fp8_case(spec, seed=31)
    ks = torch.full_like(ks, 2.0 ** -5)
    vs = torch.full_like(vs, 2.0 ** 3)
    table = torch.tensor(oracle_mod.e4m3_table())
    kd = (table[k8.long()] * 2.0 ** -5).to(torch.bfloat16)
    vd = (table[v8.long()] * 2.0 ** 3).to(torch.bfloat16)
    assert torch.equal(kd.double().nan_to_num(7.0), (table[k8.long()] * 2.0 ** -5).nan_to_num(7.0))
    d = _wdict(w)
    got = oracle_mod.decode_fp8(q, k8, v8, ks, vs, ln, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    ref = _run(oracle_mod, q, kd, vd, ln, d)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("spec", TINY[:6])
def test_fp8_form_equals_sdpa_on_dequantised_values(spec, oracle_mod):
    """Arbitrary per-(sequence, KV head) scales: the FP8 form equals torch SDPA
    (float64) over the dequantised cache, to 1e-12."""
    w, q, k8, v8, ks, vs, ln = _fp8_case(spec, seed=32)
    table = torch.tensor(oracle_mod.e4m3_table())
    kd = table[k8.long()] * ks.double()[:, :, None, None]
    vd = table[v8.long()] * vs.double()[:, :, None, None]
    got = oracle_mod.decode_fp8(q, k8, v8, ks, vs, ln, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    assert np.isfinite(got).all()  # the NaN codes sit outside the band
    G = w.NH // w.NKV
    for b in range(w.B):
        L = int(ln[b])
        if L == 0:
            assert not got[b].any()
            continue
        keep = min(w.window if w.window > 0 else w.capacity, w.capacity)
        pos = torch.arange(max(0, L - keep), L)
        kk = kd[b][:, pos % w.capacity].repeat_interleave(G, dim=0)
        vv = vd[b][:, pos % w.capacity].repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q[b].double().unsqueeze(1), kk, vv, scale=w.scale)
        np.testing.assert_allclose(got[b], o[:, 0].numpy(), rtol=0, atol=1e-12)
