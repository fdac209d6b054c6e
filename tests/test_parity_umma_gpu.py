"""GPU parity of the tcgen05 / tensor-memory split kernel (FD_PATH_UMMA)
against the FP64 oracle, through the C ABI.

The path serves the MQA geometry of "Hand-Writing Gemma 4 Flash-Decoding + an
FP4 Matvec Bonus (Part 2)" (section "One KV head breaks the textbook": one KV
head, 16 query rows, head dim 512) with no window. Fixtures cover its tile
edges (128-position tiles, 8-row tail boxes), split counts, fewer than 16 query
rows, empty and ragged sequences, a length beyond the capacity (the whole
cache, walked in slot order), NaN inside and outside the band, graph replay,
and the full-size MQA workloads; the same NaN-filled outputs, canaries and
NaN-filled workspace as the other GPU suites.
"""

import numpy as np
import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import WORKLOADS, Workload, make_inputs
from harness import check, oracle_ref, run

pytestmark = pytest.mark.gpu

W = Workload
UMMA = fd.FD_PATH_UMMA

FIXTURES = [
    W("u_len1", 1, 16, 1, 512, 64, 0, lens=(1,), seed=61),
    W("u_len7", 1, 16, 1, 512, 64, 0, lens=(7,), seed=62),
    W("u_tile_minus1", 1, 16, 1, 512, 512, 0, lens=(127,), seed=63),
    W("u_tile_exact", 1, 16, 1, 512, 512, 0, lens=(128,), seed=64),
    W("u_tile_plus1", 1, 16, 1, 512, 512, 0, lens=(129,), seed=65),
    W("u_two_tiles_ragged", 2, 16, 1, 512, 600, 0, lens=(255, 300), seed=66),
    W("u_many_tiles", 1, 16, 1, 512, 4096, 0, lens=(4000,), seed=67),
    W("u_g12", 1, 12, 1, 512, 1000, 0, lens=(999,), seed=68),
    W("u_g9_two_kv", 2, 18, 2, 512, 700, 0, lens=(650, 13), seed=69),
    W("u_batch_with_empty", 4, 16, 1, 512, 512, 0, lens=(0, 1, 17, 300), seed=70),
    W("u_len_beyond_capacity", 1, 16, 1, 512, 256, 0, lens=(1000,), seed=71),
]


def _umma_run(w, q, k, v, lens, splits=0, **kw):
    res = run(w, q, k, v, lens, splits=splits, path=UMMA, **kw)
    assert res["plan"].path == UMMA
    return res


@pytest.mark.parametrize("w", FIXTURES, ids=[f.name for f in FIXTURES])
def test_umma_fixture_matches_oracle(w):
    q, k, v, lens = make_inputs(w)
    res = _umma_run(w, q, k, v, lens)
    expect_err = fd.FD_DEVERR_LEN_CLAMPED if max(w.lens) > w.capacity else 0
    assert res["deverr"] == expect_err
    check(res, oracle_ref(w, q, k, v, lens), what=w.name)


@pytest.mark.parametrize("name", ["u_two_tiles_ragged", "u_many_tiles", "u_g9_two_kv"])
def test_umma_result_independent_of_split_count(name):
    w = next(f for f in FIXTURES if f.name == name)
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    for s in (1, 2, 3, 7, 33, 152):
        check(_umma_run(w, q, k, v, lens, splits=s), ref, what=f"{name} S={s}")


def test_umma_equals_mma_path_within_tolerance():
    """The two tensor-core families agree with each other as they do with the
    oracle (same inputs, same plan split count)."""
    w = next(f for f in FIXTURES if f.name == "u_many_tiles")
    q, k, v, lens = make_inputs(w)
    a = _umma_run(w, q, k, v, lens, splits=16)
    b = run(w, q, k, v, lens, splits=16, path=fd.FD_PATH_TC)
    assert np.abs(a["out32"].double().numpy() - b["out32"].double().numpy()).max() <= 2e-3


def test_umma_single_position_returns_v():
    w = W("u_one", 2, 16, 1, 512, 64, 0, lens=(1, 1), seed=72)
    q, k, v, lens = make_inputs(w)
    res = _umma_run(w, q, k, v, lens)
    for b in range(w.B):
        want = v[b, 0, 0].float()
        for h in range(w.NH):
            assert torch.equal(res["out32"][b, h], want)  # weight exactly 1, V exact in fp32


def test_umma_nan_inside_band_reaches_its_rows_only_through_v_dim():
    w = W("u_nan", 1, 16, 1, 512, 512, 0, lens=(300,), seed=73)
    q, k, v, lens = make_inputs(w)
    v[0, 0, 200, 7] = float("nan")
    res = _umma_run(w, q, k, v, lens)
    out = res["out32"][0]
    assert torch.isnan(out[:, 7]).all()
    out[:, 7] = 0
    assert torch.isfinite(out).all()


def test_umma_graph_replay_equals_direct_launch():
    """A CUDA-graph replay of the call gives the direct launch's bits, and
    those match the oracle."""
    w = W("u_graph", 1, 16, 1, 512, 2048, 0, lens=(1500,), seed=74)
    q, k, v, lens = make_inputs(w)
    direct = _umma_run(w, q, k, v, lens)
    check(direct, oracle_ref(w, q, k, v, lens), what="direct")
    dev = torch.device("cuda")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    fd.fd_plan_override(plan, 0, UMMA)
    ws = torch.zeros(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    out_g = torch.full_like(qd, float("nan"))
    with torch.cuda.graph(g, stream=s):
        fd.fd_decode_attn_ex(plan, ws, plan.workspace_bytes, None, qd, kd, vd, out_g, ld, w.B, w.NH, w.NKV, w.HS,
                             w.capacity, w.window, w.scale, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g.cpu().view(torch.int16), direct["out"].view(torch.int16))


def test_umma_refuses_other_shapes():
    for args in [(1, 16, 8, 256, 64, 0), (1, 16, 2, 512, 64, 0), (1, 16, 1, 512, 64, 32)]:
        p = fd.fd_plan(*args, 0)
        with pytest.raises(fd.FdError):
            fd.fd_plan_override(p, 0, UMMA)


@pytest.mark.parametrize("name", ["gemma_global_mqa_4k", "gemma_global_mqa_32k", "gemma_mqa_long"])
def test_umma_full_size_workload_sampled_rows(name):
    from test_parity_gpu import _sample_rows
    w = WORKLOADS[name]
    dev = torch.device("cuda")
    q, k, v, lens = make_inputs(w, device=dev)
    res = _umma_run(w, q, k, v, lens, inputs_on_device=True)
    assert torch.isfinite(res["out32"]).all(), "NaN/inf in some row"
    assert res["deverr"] == 0
    rows = _sample_rows(w, lens)
    qh, kh, vh = q.cpu(), k.cpu(), v.cpu()
    del q, k, v
    torch.cuda.empty_cache()
    check(res, oracle_ref(w, qh, kh, vh, lens, rows=rows), rows=rows, what=name)


def test_umma_rising_scores_rescale_across_tiles():
    """Scores that grow tile after tile by more than the 2^8 the running
    maximum may lag behind: the rescale of O in tensor memory runs at several
    tile boundaries, and at S = 1 one block sees them all."""
    w = W("u_rising", 1, 16, 1, 512, 1024, 0, lens=(1000,), seed=75)
    q, k, v, lens = make_inputs(w)
    ramp = torch.linspace(0.2, 6.0, w.capacity).view(1, 1, -1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    ref = oracle_ref(w, q, k, v, lens)
    for s in (1, 3):
        check(_umma_run(w, q, k, v, lens, splits=s), ref, what=f"rising S={s}")


def test_umma_nan_key_in_a_middle_tile_reaches_every_row():
    w = W("u_nan_k", 1, 16, 1, 512, 1024, 0, lens=(900,), seed=76)
    q, k, v, lens = make_inputs(w)
    k[0, 0, 400, 3] = float("nan")
    res = _umma_run(w, q, k, v, lens, splits=1)
    assert torch.isnan(res["out32"][0]).all()
    res = _umma_run(w, q, k, v, lens, splits=4)
    assert torch.isnan(res["out32"][0]).all()


@pytest.mark.parametrize("splits", [1, 5, 40])
def test_umma_min_len_bound_kept_and_broken(splits):
    """The tcgen05 kernel reads nothing before a sequence's length arrives, so
    the plan's lower bound on the lengths changes no result: kept, the output
    is bit-identical to the plan without it and no error bit is set; broken,
    the output is still exact and FD_DEVERR_MIN_LEN is raised."""
    w = Workload("u_min_len", 2, 16, 1, 512, 2048, 0, lens=(1500, 700), seed=72)
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    base = _umma_run(w, q, k, v, lens, splits=splits)
    kept = _umma_run(w, q, k, v, lens, splits=splits, min_len=700)
    check(kept, ref, what=f"umma min_len kept S={splits}")
    assert kept["deverr"] == 0
    assert torch.equal(kept["out32"], base["out32"])
    broken = _umma_run(w, q, k, v, lens, splits=splits, min_len=1024)
    check(broken, ref, what=f"umma min_len broken S={splits}")
    assert broken["deverr"] & fd.FD_DEVERR_MIN_LEN


def test_umma_chunks_are_whole_16_position_steps():
    """Plans for the tcgen05 kernel round chunks to 16 positions: every split
    but the band's last ends on a P.V step, and results do not depend on the
    split count even where a chunk of 1 position would have been asked for."""
    w = Workload("u_granule", 1, 16, 1, 512, 4096, 0, lens=(1000,), seed=73)
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    outs = []
    for splits in (7, 63, 152, 1000):
        res = _umma_run(w, q, k, v, lens, splits=splits)
        assert res["plan"].granule == 16
        check(res, ref, what=f"umma granule S={splits}")
        outs.append(res["out32"])
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2e-3
