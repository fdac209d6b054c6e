"""GPU parity of libfd.so against the FP64 oracle, through the C ABI.

Fixture categories follow "Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec
Bonus (Part 2)", section "The test that catches what parity misses": split
boundaries, pre-window positions, ring wrap, batch > 1; every cache slot
outside the live band holds NaN, every output buffer is guarded by canaries,
and the workspace starts filled with NaN bytes so an unwritten partial would
surface.
"""

import numpy as np
import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import WORKLOADS, Workload, make_inputs
from harness import Guarded, check, oracle_ref, run

pytestmark = pytest.mark.gpu

W = Workload

FIXTURES = [
    # ---- split boundaries (band vs tile / chunk edges)
    W("band1_mqa", 1, 16, 1, 512, 64, 0, lens=(1,), seed=1),
    W("band2_ring", 1, 16, 8, 256, 64, 0, lens=(2,), seed=2),
    W("tile_minus1_d256", 1, 16, 8, 256, 64, 0, lens=(31,), seed=3),
    W("tile_exact_d256", 1, 16, 8, 256, 64, 0, lens=(32,), seed=4),
    W("tile_plus1_d256", 1, 16, 8, 256, 64, 0, lens=(33,), seed=5),
    W("tile_pm1_d512", 2, 16, 1, 512, 64, 0, lens=(15, 17), seed=6),
    W("tile_pm1_d128", 2, 32, 8, 128, 128, 0, lens=(47, 49), seed=7),
    W("tile_pm1_d64", 2, 8, 8, 64, 256, 0, lens=(95, 97), seed=8),
    # ---- pre-window positions
    W("len_below_window", 1, 16, 8, 256, 64, 48, lens=(40,), seed=9),
    W("len_equal_window", 1, 16, 8, 256, 64, 48, lens=(48,), seed=10),
    W("len_window_plus1", 1, 16, 8, 256, 64, 48, lens=(49,), seed=11),
    W("lo_not_tile_aligned", 1, 16, 1, 512, 128, 37, lens=(100,), seed=12),
    # ---- ring wrap
    W("ring_full_1024", 1, 16, 8, 256, 1024, 1024, lens=(1024,), seed=13),
    W("ring_wrap_1025", 1, 16, 8, 256, 1024, 1024, lens=(1025,), seed=14),
    W("ring_wrap_32x", 1, 16, 8, 256, 1024, 1024, lens=(32768,), seed=15),
    W("ring_wrap_33000", 1, 16, 8, 256, 1024, 1024, lens=(33000,), seed=16),
    W("ring_dead_slots_w1000", 1, 16, 8, 256, 1024, 1000, lens=(5000,), seed=17),
    W("ring_straddles_slot0", 1, 16, 8, 256, 64, 64, lens=(100,), seed=18),
    # ---- batch > 1
    W("batch16_ragged_llama", 16, 32, 8, 128, 512, 0,
      lens=(1, 512, 17, 300, 2, 511, 64, 65, 128, 129, 250, 3, 400, 33, 90, 256), seed=19),
    W("batch4_mqa_with_empty", 4, 16, 1, 512, 512, 0, lens=(0, 1, 17, 300), seed=20),
    W("batch3_ring_mixed", 3, 16, 8, 256, 128, 100, lens=(0, 99, 1000), seed=21),
    # ---- other groupings and head sizes
    W("mha_d64", 2, 8, 8, 64, 200, 0, lens=(200, 77), seed=22),
    W("g8_d128", 1, 16, 2, 128, 300, 0, lens=(300,), seed=23),
    W("g16_d64", 1, 16, 1, 64, 300, 0, lens=(299,), seed=24),
    W("g4_d512", 1, 8, 2, 512, 200, 0, lens=(150,), seed=25),
    W("g2_d128_window1", 2, 16, 8, 128, 64, 1, lens=(37, 1), seed=26),
]


@pytest.mark.parametrize("path", [fd.FD_PATH_TC, fd.FD_PATH_SIMT], ids=["tc", "simt"])
@pytest.mark.parametrize("w", FIXTURES, ids=[f.name for f in FIXTURES])
def test_fixture_matches_oracle(w, path):
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    res = run(w, q, k, v, lens, path=path)
    check(res, ref, what=w.name)
    assert res["deverr"] == 0


SPLIT_CASES = [
    W("split_mqa", 2, 16, 1, 512, 700, 0, lens=(700, 333), seed=31),
    W("split_ring", 1, 16, 8, 256, 256, 200, lens=(1234,), seed=32),
    W("split_llama", 3, 32, 8, 128, 400, 0, lens=(400, 1, 123), seed=33),
]


@pytest.mark.parametrize("w", SPLIT_CASES, ids=[c.name for c in SPLIT_CASES])
def test_result_independent_of_split_count(w):
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    band = max(min(int(x), w.window if w.window > 0 else w.capacity) for x in lens)
    outs = []
    for s in sorted({1, 2, 3, 7, 64, band, band + 5}):
        res = run(w, q, k, v, lens, splits=s, cluster=1)
        check(res, ref, what=f"{w.name} S={s}")
        outs.append(res["out32"])
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2e-3


FUSED_CASES = [
    W("fu_ring", 1, 16, 8, 256, 1024, 1024, lens=(32768,), seed=71),
    W("fu_llama_batch", 5, 32, 8, 128, 600, 0, lens=(600, 0, 1, 299, 64), seed=72),
    W("fu_g8_d512", 2, 16, 2, 512, 300, 0, lens=(300, 17), seed=73),
]


@pytest.mark.parametrize("w", FUSED_CASES, ids=[c.name for c in FUSED_CASES])
def test_fused_merge_equals_merge_kernel(w):
    """The last split block of each group merging the partials itself (no merge
    kernel) agrees with the oracle and with the separate merge kernel, for split
    counts from 2 up to the fused limit; the counters are back at zero after
    every call."""
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    G = w.NH // w.NKV
    s_max = (256 << 10) // (G * w.HS * 4)  # the group's partials within 256 KB
    for S in sorted(x for x in {2, 3, 8, 19, 38, s_max} if x <= s_max):
        outs = {}
        for fused in (0, 1):
            res = run(w, q, k, v, lens, splits=S, cluster=1, fused=fused)
            assert res["plan"].fused == fused
            check(res, ref, what=f"{w.name} S={S} fused={fused}")
            outs[fused] = res["out32"]
        assert (outs[0] - outs[1]).abs().max().item() <= 1e-5


GROUP_CASES = FUSED_CASES + [
    W("gs_mqa_many_splits", 1, 16, 1, 512, 32768, 0, lens=(20000,), seed=74),
    W("gs_llama_tiny", 1, 32, 8, 128, 512, 0, lens=(256,), seed=75),
    W("gs_ring_not_full", 1, 16, 8, 256, 1024, 1024, lens=(700,), seed=76),
    W("gs_window_chunks", 2, 16, 8, 256, 1024, 300, lens=(5000, 299), seed=77),
]


@pytest.mark.parametrize("w", GROUP_CASES, ids=[c.name for c in GROUP_CASES])
def test_group_step_merge_matches_oracle_and_merge_kernel(w):
    """fused = 2: every split block of a group waits for the group inside the
    (cooperative) split launch, then merges a share of the outputs. Agrees with
    the oracle and with the merge kernel at every split count the grid allows
    (one wave), is bit-identical run to run, and leaves both counter words at
    zero."""
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    s_cap = plan.num_sms * plan.ctas_per_sm // (w.B * w.NKV)
    assert s_cap >= 2
    for S in sorted(x for x in {2, 3, 8, 19, 32, 38, 76, s_cap} if x <= s_cap):
        base = run(w, q, k, v, lens, splits=S, cluster=1, fused=0)
        res = run(w, q, k, v, lens, splits=S, cluster=1, fused=2)
        assert res["plan"].fused == 2
        assert res["plan"].workspace_zero_bytes >= 2 * 4 * w.B * w.NKV
        check(res, ref, what=f"{w.name} S={S} group step")
        assert res["deverr"] & fd.FD_DEVERR_WAIT_TIMEOUT == 0
        assert (res["out32"] - base["out32"]).abs().max().item() <= 1e-5
        again = run(w, q, k, v, lens, splits=S, cluster=1, fused=2)
        assert torch.equal(again["out32"], res["out32"])
    with pytest.raises(fd.FdError):  # a grid beyond one wave cannot wait on itself
        fd.fd_plan_override(fd.fd_plan_t.from_buffer_copy(plan), s_cap + 1, 0, 1, 2)


def test_group_step_with_min_len_bound():
    """The group step behind early reads: with the plan's lower bound on the
    lengths kept, the result equals the plan without it; broken, it is still
    exact and FD_DEVERR_MIN_LEN is raised; the counter words are zero after
    both."""
    w = W("gs_min_len", 1, 16, 8, 256, 1024, 1024, lens=(700,), seed=79)
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    S = min(16, plan.num_sms * plan.ctas_per_sm // (w.B * w.NKV))  # one wave
    base = run(w, q, k, v, lens, splits=S, cluster=1, fused=2)
    kept = run(w, q, k, v, lens, splits=S, cluster=1, fused=2, min_len=700)
    check(kept, ref, what="group step, min_len kept")
    assert kept["deverr"] == 0 and torch.equal(kept["out32"], base["out32"])
    broken = run(w, q, k, v, lens, splits=S, cluster=1, fused=2, min_len=1024)
    check(broken, ref, what="group step, min_len broken")
    assert broken["deverr"] & fd.FD_DEVERR_MIN_LEN


def test_group_step_graph_replays_reuse_the_counters():
    """A captured group-step call replayed with new lengths: every replay is
    exact (the counter words return to zero each time), and the E4M3 cache
    takes the same step."""
    w = W("gs_graph", 1, 16, 8, 256, 1024, 1024, lens=(5000,), seed=78)
    q, k, v, lens = make_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    fd.fd_plan_override(plan, 0, 0, 1, 2)
    assert plan.fused == 2
    ws = torch.zeros(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    o16 = Guarded(w.B * w.NH * w.HS * 2, dev, fill=0xFF)
    o32 = Guarded(w.B * w.NH * w.HS * 4, dev, fill=0xFF)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture
        fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, o32.ptr(), qd, kd, vd, o16.ptr(), ld, w.B, w.NH,
                             w.NKV, w.HS, w.capacity, w.window, w.scale)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):  # three calls in a row on one workspace
            fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, o32.ptr(), qd, kd, vd, o16.ptr(), ld, w.B,
                                 w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    fd.fd_get_device_error()
    for new_len in (3000, 1024, 700, 1, 5000):
        ld.fill_(new_len)
        g.replay()
        torch.cuda.synchronize()
        res = dict(out=o16.view(torch.bfloat16, (w.B, w.NH, w.HS)).cpu(),
                   out32=o32.view(torch.float32, (w.B, w.NH, w.HS)).cpu(),
                   counters_zero=bool((ws[: plan.workspace_zero_bytes] == 0).all().item()),
                   canaries=o16.canaries_intact() and o32.canaries_intact())
        check(res, oracle_ref(w, q, k, v, torch.tensor([new_len], dtype=torch.int32)),
              what=f"group step replay, len {new_len}")
    assert fd.fd_get_device_error() == 0


@pytest.mark.parametrize("hs,nh,nkv", [(256, 16, 8), (128, 32, 8), (512, 16, 1)], ids=["d256", "d128", "d512"])
def test_lengths_beyond_the_plan_bound_stay_exact(hs, nh, nkv):
    """A plan sized for short bands (max_len = 128: whole-tile splits, and for
    the sliding-ring tile its one-stage form, each split one tile) called with
    far longer bands: the device divides each band itself, so every split just
    takes several tiles through its stages and the result stays exact."""
    w = W(f"beyond_d{hs}", 2, nh, nkv, hs, 2048, 0, lens=(2000, 700), seed=80 + hs)
    q, k, v, lens = make_inputs(w)
    res = run(w, q, k, v, lens, max_len=128)
    assert res["plan"].max_band == 128 and res["plan"].granule > 1
    check(res, oracle_ref(w, q, k, v, lens), what=f"d{hs} lens beyond max_len")


CLUSTER_CASES = [
    W("cl_mqa", 2, 16, 1, 512, 700, 0, lens=(700, 3), seed=61),
    W("cl_ring", 1, 16, 8, 256, 256, 200, lens=(1234,), seed=62),
    W("cl_llama", 3, 32, 8, 128, 400, 0, lens=(400, 1, 0), seed=63),
    W("cl_g16_d64", 1, 16, 1, 64, 300, 0, lens=(299,), seed=64),
]


@pytest.mark.parametrize("w", CLUSTER_CASES, ids=[c.name for c in CLUSTER_CASES])
def test_result_independent_of_cluster_size(w):
    """Thread-block clusters that combine partials in distributed shared
    memory, with one cluster per band (direct output) or several (merged
    partials), agree with the oracle for every cluster size."""
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    maxc = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window).max_cluster
    for cluster in (1, 2, 4, 8, 16):
        if cluster > maxc or (w.HS // cluster) % 4:
            continue
        for splits in sorted({cluster, 2 * cluster, 3 * cluster, 8 * cluster}):
            res = run(w, q, k, v, lens, splits=splits, cluster=cluster)
            check(res, ref, what=f"{w.name} S={splits} cluster={cluster}")
            assert res["deverr"] == 0


def test_single_position_band_returns_v_exactly():
    for w, slot in [(W("len1", 1, 16, 8, 256, 64, 0, lens=(1,), seed=41), 0),
                    (W("win1", 1, 16, 1, 512, 64, 1, lens=(150,), seed=42), 149 % 64)]:
        q, k, v, lens = make_inputs(w)
        for path in (fd.FD_PATH_TC, fd.FD_PATH_SIMT):
            for splits in (0, 1, 5):
                res = run(w, q, k, v, lens, splits=splits, path=path, cluster=1 if splits else 0)
                G = w.NH // w.NKV
                for h in range(w.NH):
                    vrow = v[0, h // G, slot]
                    assert torch.equal(res["out32"][0, h], vrow.float()), (w.name, path, splits, h)
                    assert torch.equal(res["out"][0, h].view(torch.int16), vrow.view(torch.int16))


def test_nan_inside_band_reaches_only_its_group():
    w = W("nan_in_band", 1, 16, 8, 256, 256, 0, lens=(200,), seed=43)
    q, k, v, lens = make_inputs(w)
    k = k.clone()
    k[0, 3, 77, 10] = float("nan")
    res = run(w, q, k, v, lens)
    o = res["out32"][0]
    G = 2
    assert torch.isnan(o[3 * G:4 * G]).all()
    rest = torch.cat([o[:3 * G], o[4 * G:]])
    assert torch.isfinite(rest).all()


def test_repeat_runs_are_bitwise_identical():
    w = W("determinism", 2, 16, 1, 512, 2048, 0, lens=(2048, 1111), seed=44)
    q, k, v, lens = make_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    first = None
    for _ in range(100):
        out = torch.empty_like(qd)
        fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, None, qd, kd, vd, out, ld, w.B, w.NH, w.NKV,
                             w.HS, w.capacity, w.window, w.scale)
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))


def test_library_workspace_entry_equals_explicit_and_graph_replay():
    """fd_decode_attn (library-owned workspace) == fd_decode_attn_ex, and a CUDA
    graph replay of the call == the direct launch, bit for bit (the graph-parity
    contract of SharpInference issue #156, Work Item B)."""
    w = W("graph", 1, 16, 8, 256, 1024, 1024, lens=(5000,), seed=45)
    q, k, v, lens = make_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    res = run(w, q, k, v, lens)
    s = torch.cuda.Stream()
    out = torch.empty_like(qd)
    with torch.cuda.stream(s):
        fd.fd_decode_attn(qd, kd, vd, out, ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)  # warm-up
    s.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), res["out"].view(torch.int16))
    g = torch.cuda.CUDAGraph()
    out_g = torch.zeros_like(qd)
    with torch.cuda.graph(g, stream=s):
        fd.fd_decode_attn(qd, kd, vd, out_g, ld, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g.view(torch.int16), out.view(torch.int16))
    # lens live on the device: a replay sees new lengths. The same capture
    # through fd_decode_attn_ex with the fp32 copy, checked against the
    # oracle at the full tolerance after each replay.
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    ws = torch.zeros(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    o16 = Guarded(w.B * w.NH * w.HS * 2, dev, fill=0xFF)
    o32 = Guarded(w.B * w.NH * w.HS * 4, dev, fill=0xFF)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, o32.ptr(), qd, kd, vd, o16.ptr(), ld, w.B, w.NH,
                             w.NKV, w.HS, w.capacity, w.window, w.scale)
    for new_len in (3000, 1024, 700, 5000):
        ld.fill_(new_len)
        g.replay()
        g2.replay()
        torch.cuda.synchronize()
        res2 = dict(out=o16.view(torch.bfloat16, (w.B, w.NH, w.HS)).cpu(),
                    out32=o32.view(torch.float32, (w.B, w.NH, w.HS)).cpu(), counters_zero=True,
                    canaries=o16.canaries_intact() and o32.canaries_intact())
        ref2 = oracle_ref(w, q, k, v, torch.tensor([new_len], dtype=torch.int32))
        check(res2, ref2, what=f"graph replay with len {new_len}")
        assert torch.equal(out_g.cpu().view(torch.int16), res2["out"].view(torch.int16))


def test_device_error_word_reports_repaired_lengths():
    w = W("deverr", 2, 16, 8, 256, 64, 0, lens=(10, 10), seed=46)
    q, k, v, _ = make_inputs(w, poison=False)
    # negative length -> treated as 0 (zero output), flagged
    res = run(w, q, k, v, torch.tensor([-5, 10], dtype=torch.int32))
    assert res["deverr"] & fd.FD_DEVERR_LEN_NEGATIVE
    assert torch.equal(res["out32"][0], torch.zeros_like(res["out32"][0]))
    # no window, len > capacity -> the last `capacity` positions, flagged
    lens = torch.tensor([150, 64], dtype=torch.int32)
    res = run(w, q, k, v, lens)
    assert res["deverr"] & fd.FD_DEVERR_LEN_CLAMPED
    w2 = W("deverr_w", 2, 16, 8, 256, 64, 64, lens=(150, 64), seed=46)
    res2 = run(w2, q, k, v, lens)
    assert res2["deverr"] == 0
    assert torch.equal(res["out32"], res2["out32"])


def test_bad_arguments_launch_nothing():
    w = WORKLOADS["llama_tiny"]
    q, k, v, lens = make_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    out = torch.full_like(qd, 7.0)
    with pytest.raises(fd.FdError) as e:
        fd.fd_decode_attn(qd, kd, vd, out, ld, w.B, w.NH, w.NKV, 96, w.capacity, w.window, w.scale)
    assert e.value.status == fd.FD_ERR_UNSUPPORTED
    raw = torch.empty(qd.numel() * 2 + 2, dtype=torch.uint8, device=dev)
    with pytest.raises(fd.FdError) as e:
        fd.fd_decode_attn(raw.data_ptr() + 2, kd, vd, out, ld, w.B, w.NH, w.NKV, w.HS, w.capacity,
                          w.window, w.scale)
    assert e.value.status == fd.FD_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert (out == 7.0).all()


# --------------------------------------------------- full-size workloads

def _sample_rows(w, lens, n=8, seed=0):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (w.B - 1, w.NH - 1)}
    if w.B > 1:
        L = lens.numpy()
        rows |= {(int(L.argmin()), 0), (int(L.argmax()), w.NH // 2)}
    while len(rows) < min(n, w.B * w.NH):
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.NH))))
    return sorted(rows)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload_sampled_rows(name):
    """Full sizes in the launch configuration the benchmark times (fd_plan for
    the device, max_len <= 0), inputs drawn on the device; the oracle checks a
    sample of (sequence, head) rows, and every row is checked for finiteness
    (the NaN poison outside the band)."""
    w = WORKLOADS[name]
    dev = torch.device("cuda")
    q, k, v, lens = make_inputs(w, device=dev)
    res = run(w, q, k, v, lens, inputs_on_device=True)
    assert torch.isfinite(res["out32"]).all(), "NaN/inf in some row"
    assert res["deverr"] == 0
    rows = _sample_rows(w, lens)
    qh, kh, vh = q.cpu(), k.cpu(), v.cpu()
    del q, k, v
    torch.cuda.empty_cache()
    ref = oracle_ref(w, qh, kh, vh, lens, rows=rows)
    check(res, ref, rows=rows, what=name)


@pytest.mark.parametrize("q_mul", [64.0, 1e-4], ids=["peaked", "flat"])
def test_extreme_score_scales_match_oracle(q_mul):
    """Very peaked (scores in the hundreds) and nearly flat softmaxes, on both
    kernel families: the max shift and the hi/lo P split keep the tolerance."""
    w = W("extreme", 2, 16, 8, 128, 400, 0, lens=(400, 133), seed=48)
    q, k, v, lens = make_inputs(w)
    q = (q.float() * q_mul).to(torch.bfloat16)
    ref = oracle_ref(w, q, k, v, lens)
    for path in (fd.FD_PATH_TC, fd.FD_PATH_SIMT):
        check(run(w, q, k, v, lens, path=path), ref, what=f"q x {q_mul} path {path}")


@pytest.mark.parametrize("B", [64, 200], ids=["B64_longest_first", "B200_natural_order"])
def test_large_batches_around_the_ordering_cutoff(B):
    """Batches at the longest-band-first limit (64 sequences) and above it
    (blocks in natural order), with empty sequences and lengths beyond the
    capacity (no window: the band is clamped and flagged)."""
    rng = np.random.default_rng(B)
    lens = tuple(int(x) for x in rng.integers(0, 41, size=B))
    w = W(f"batch{B}", B, 8, 8, 64, 32, 0, lens=lens, seed=49 + B)
    q, k, v, ln = make_inputs(w)
    ref = oracle_ref(w, q, k, v, ln)
    for path in (fd.FD_PATH_TC, fd.FD_PATH_SIMT):
        res = run(w, q, k, v, ln, path=path)
        assert res["deverr"] == (fd.FD_DEVERR_LEN_CLAMPED if max(lens) > 32 else 0)
        check(res, ref, what=f"B={B} path {path}")


@pytest.mark.parametrize("splits", [2, 257, 600])
def test_staged_merge_with_many_partials(splits):
    """64 or more rows (B * NH) take the staged merge (partials brought into
    shared memory 256 slots per stage): one, two and three stages, an empty
    sequence (all partials empty: zero rows) and sequences shorter than the
    split count (empty partials past their active splits)."""
    w = W("staged_merge", 4, 16, 2, 128, 1200, 0, lens=(1200, 700, 0, 5), seed=91)
    assert w.B * w.NH >= 64
    q, k, v, lens = make_inputs(w)
    res = run(w, q, k, v, lens, splits=splits)
    assert res["plan"].num_splits == splits and res["deverr"] == 0
    check(res, oracle_ref(w, q, k, v, lens), what=f"S={splits}")
    assert torch.equal(res["out32"][2], torch.zeros_like(res["out32"][2]))


def test_staged_merge_nan_in_scores_reaches_only_its_group():
    """A NaN key makes every row of its group NaN through the partials' m and
    l; the other group and the other sequences stay finite (staged merge)."""
    w = W("staged_nan", 4, 16, 2, 128, 300, 0, lens=(300, 200, 1, 77), seed=92)
    q, k, v, lens = make_inputs(w)
    k[1, 1, 150, 3] = float("nan")
    res = run(w, q, k, v, lens, splits=9)
    G = w.NH // w.NKV
    out = res["out32"]
    assert torch.isnan(out[1, G:]).all()
    assert torch.isfinite(out[1, :G]).all() and torch.isfinite(out[[0, 2, 3]]).all()


@pytest.mark.parametrize("lens", [(0,), (1,), (100,), (1023,), (1024,), (5000,)])
@pytest.mark.parametrize("splits", [0, 1, 7, 32])
def test_ring_first_tile_copied_before_the_length(lens, splits):
    """A ring (window == capacity) with one sequence: each split block copies
    its first tile for a full ring before it knows the length. A ring that is
    not full (len < capacity) drops those copies: empty slices (which wait for
    them before leaving), partial slices, one split (the output written
    directly) and len == 0 all match the oracle; full rings use the copies."""
    w = W("ring_spec", 1, 16, 8, 256, 1024, 1024, lens=lens, seed=93)
    q, k, v, lens_t = make_inputs(w)
    res = run(w, q, k, v, lens_t, splits=splits)
    assert res["deverr"] == 0
    check(res, oracle_ref(w, q, k, v, lens_t), what=f"len={lens[0]} S={splits}")
