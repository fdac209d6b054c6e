"""GPU parity of the FP8 (E4M3) cache path of libfd.so against the FP64 oracle,
through the C ABI.

The cache form follows "Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec
Bonus (Part 2)": the open-problem paragraph just before "What we'd tell the
next person" leaves the long-band latency residual to FP8 KV storage, and that
section says FP8 KV is widened inline where it is used. Reading taken: E4M3
codes with one fp32 scale per (sequence, KV head) for K and for V. The
fixtures are the bf16 suite's (split boundaries, pre-window positions, ring
wrap, batch > 1, other groupings); every dead slot holds the E4M3 NaN code,
outputs are guarded by canaries and the workspace starts as NaN bytes.
Tolerances are the bf16 suite's.
"""

import numpy as np
import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import E4M3_NAN_CODE, WORKLOADS, make_inputs_fp8
from harness import check, oracle_ref_fp8, run_fp8
from test_parity_gpu import FIXTURES, W, _sample_rows

pytestmark = pytest.mark.gpu

FP8_EXTRA = [
    # odd group sizes and every head size at a partial last tile
    W("fp8_g1_d128", 2, 8, 8, 128, 300, 0, lens=(300, 5), seed=41),
    W("fp8_g16_d256", 1, 32, 2, 256, 500, 0, lens=(417,), seed=42),
    W("fp8_g12_d512", 1, 12, 1, 512, 700, 0, lens=(699,), seed=43),
]


@pytest.mark.parametrize("w", FIXTURES + FP8_EXTRA, ids=[f.name for f in FIXTURES + FP8_EXTRA])
def test_fp8_fixture_matches_oracle(w):
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    res = run_fp8(w, q, k8, v8, ks, vs, lens)
    assert res["deverr"] == 0
    check(res, oracle_ref_fp8(w, q, k8, v8, ks, vs, lens), what=w.name)


@pytest.mark.parametrize("name", ["tile_pm1_d512", "ring_wrap_33000", "batch16_ragged_llama"])
def test_fp8_result_independent_of_split_count(name):
    w = next(f for f in FIXTURES if f.name == name)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    ref = oracle_ref_fp8(w, q, k8, v8, ks, vs, lens)
    for s in (1, 2, 3, 7, 64):
        check(run_fp8(w, q, k8, v8, ks, vs, lens, splits=s), ref, what=f"{name} S={s}")


def test_fp8_fused_merge_and_clusters_agree_with_the_oracle():
    w = next(f for f in FIXTURES if f.name == "ring_wrap_1025")
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    ref = oracle_ref_fp8(w, q, k8, v8, ks, vs, lens)
    check(run_fp8(w, q, k8, v8, ks, vs, lens, splits=8, fused=1), ref, what="fused")
    for S in (2, 8, 32):
        res = run_fp8(w, q, k8, v8, ks, vs, lens, splits=S, fused=2)
        assert res["plan"].fused == 2
        check(res, ref, what=f"group step S={S}")
    check(run_fp8(w, q, k8, v8, ks, vs, lens, splits=8, cluster=8), ref, what="one cluster")
    check(run_fp8(w, q, k8, v8, ks, vs, lens, splits=16, cluster=4), ref, what="clusters of 4")


def test_fp8_single_position_band_returns_scaled_v():
    """A one-position band has softmax weight exactly 1: the output is the
    dequantised V row, E4M3(code) x scale, up to one fp32 rounding."""
    w = W("fp8_one", 2, 16, 2, 256, 64, 0, lens=(1, 1), seed=44)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    res = run_fp8(w, q, k8, v8, ks, vs, lens)
    import oracle
    table = oracle.e4m3_table()
    G = w.NH // w.NKV
    for b in range(w.B):
        for h in range(w.NH):
            kvh = h // G
            want = table[v8[b, kvh, 0].numpy()] * float(vs[b, kvh])
            got = res["out32"][b, h].double().numpy()
            assert np.allclose(got, want, rtol=2 ** -23, atol=0), (b, h)


def test_fp8_nan_code_inside_band_reaches_only_its_group():
    w = W("fp8_nan", 1, 16, 2, 128, 64, 0, lens=(40,), seed=45)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    v8[0, 1, 17, 3] = E4M3_NAN_CODE  # live position of KV head 1
    res = run_fp8(w, q, k8, v8, ks, vs, lens)
    G = w.NH // w.NKV
    assert torch.isfinite(res["out32"][0, :G]).all()
    assert torch.isnan(res["out32"][0, G:, 3]).all()


def test_fp8_auto_entry_equals_explicit_and_graph_replay():
    """fd_decode_attn_fp8 (library workspace, device plan) gives the bits of
    fd_decode_attn_fp8_ex, both directly and replayed from a CUDA graph."""
    w = WORKLOADS["gemma_local_ring"]
    dev = torch.device("cuda")
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w, device=dev)
    ld = lens.to(dev)
    ref = run_fp8(w, q, k8, v8, ks, vs, lens, inputs_on_device=True)
    out = torch.empty_like(q)
    fd.fd_decode_attn_fp8(q, k8, v8, ks, vs, out, ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), ref["out"].view(torch.int16))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    out2 = torch.full_like(q, float("nan"))
    with torch.cuda.stream(s):
        fd.fd_decode_attn_fp8(q, k8, v8, ks, vs, out2, ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window,
                              w.scale, stream=s)  # workspace for this stream exists before capture
        s.synchronize()
        out2.fill_(float("nan"))
        with torch.cuda.graph(g, stream=s):
            fd.fd_decode_attn_fp8(q, k8, v8, ks, vs, out2, ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window,
                                  w.scale, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2.cpu().view(torch.int16), ref["out"].view(torch.int16))


@pytest.mark.parametrize("name", ["gemma_local_ring", "gemma_global_mqa_32k", "llama_ragged", "gemma_mqa_long"])
def test_fp8_full_size_workload_sampled_rows(name):
    """Full sizes with the device plan (the benchmark's launch configuration),
    inputs drawn and quantised on the device; sampled rows against the
    oracle, every row checked for finiteness (NaN codes fill dead slots)."""
    w = WORKLOADS[name]
    dev = torch.device("cuda")
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w, device=dev)
    res = run_fp8(w, q, k8, v8, ks, vs, lens, inputs_on_device=True)
    assert torch.isfinite(res["out32"]).all(), "NaN/inf in some row"
    assert res["deverr"] == 0
    rows = _sample_rows(w, lens)
    qh, kh, vh, ksh, vsh = q.cpu(), k8.cpu(), v8.cpu(), ks.cpu(), vs.cpu()
    del q, k8, v8
    torch.cuda.empty_cache()
    check(res, oracle_ref_fp8(w, qh, kh, vh, ksh, vsh, lens, rows=rows), rows=rows, what=name)


def test_fp8_mqa_tile_both_warp_counts():
    """The head-dim-512, 16-row E4M3 tile comes with eight consumer warps (grid
    of at most one block per SM) and with four (more blocks): both match the
    oracle."""
    w = W("fp8_mqa_warps", 2, 16, 1, 512, 3000, 0, lens=(2999, 1234), seed=46)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    ref = oracle_ref_fp8(w, q, k8, v8, ks, vs, lens)
    seen = set()
    for s in (8, 76, 100, 150):
        res = run_fp8(w, q, k8, v8, ks, vs, lens, splits=s)
        seen.add(res["plan"].consumer_warps)
        check(res, ref, what=f"S={s} warps={res['plan'].consumer_warps}")
    assert seen == {4, 8}


@pytest.mark.parametrize("q_mul,k_mul,v_mul", [(1e4, 1.0, 1.0), (1e-3, 1.0, 1.0), (1.0, 1e-3, 1e3), (30.0, 8.0, 1e-2)],
                         ids=["q_large", "q_tiny", "k_small_v_large", "peaked"])
def test_fp8_extreme_magnitudes(q_mul, k_mul, v_mul):
    """The per-block power-of-two Q scale and the folded K scale keep scores
    exact in fp32 and finite for very large / small inputs; the V scale
    multiplies O once. Checked against the oracle on the same codes and
    scales (the fp32 tolerance is relative to the output's scale here)."""
    w = W("fp8_extreme", 2, 16, 2, 256, 300, 0, lens=(300, 77), seed=47)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    q = (q.float() * q_mul).to(torch.bfloat16)
    ks, vs = ks * k_mul, vs * v_mul
    res = run_fp8(w, q, k8, v8, ks, vs, lens)
    ref = oracle_ref_fp8(w, q, k8, v8, ks, vs, lens)
    got = res["out32"].double().numpy()
    assert np.isfinite(got).all()
    tol = 2e-3 * max(1.0, v_mul)
    assert np.abs(got - ref).max() <= tol, np.abs(got - ref).max()


@pytest.mark.parametrize("length", [0, 40, 1024, 3000])
def test_fp8_ring_first_tile_copied_before_the_length(length):
    """The E4M3 ring (window == capacity): a full ring uses the first tile
    copied before the length arrived; a ring that is not full drops it."""
    w = W("fp8_ring_spec", 1, 16, 8, 256, 1024, 1024, lens=(length,), seed=48)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    for splits in (0, 5):
        res = run_fp8(w, q, k8, v8, ks, vs, lens, splits=splits)
        assert res["deverr"] == 0
        check(res, oracle_ref_fp8(w, q, k8, v8, ks, vs, lens), what=f"len={length} S={splits}")
