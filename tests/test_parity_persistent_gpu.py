"""GPU parity of the persistent split grid (fd_plan_persistent) against the
FP64 oracle and against the one-block-per-split grid, through the C ABI.

"Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section
"One KV head breaks the textbook", gives every (KV head, split) its own block;
the persistent grid runs the same work items on a fixed set of blocks that take
them from a counter in the workspace, the copy warps streaming the next item
while the MMA warps finish the current one. Each item computes exactly what its
block would have, so the outputs must be bit-identical to the per-split grid,
and within the oracle's tolerance. Grids narrowed to 1-5 blocks make every
block run many items (the item queue and the stage ring wrap many times); the
counter must be back at zero after every call (checked by the harness), also
across calls that reuse one workspace and graph replays.
"""

import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import WORKLOADS, make_inputs, make_inputs_fp8
from harness import Guarded, check, oracle_ref, oracle_ref_fp8, run, run_fp8
from test_parity_gpu import FIXTURES, W, _sample_rows

pytestmark = pytest.mark.gpu

ALL = 1 << 30  # the plan's persistent block count


def _same_bits(a, b, what=""):
    assert torch.equal(a["out"].view(torch.int16), b["out"].view(torch.int16)), f"{what}: bf16 output differs"
    assert torch.equal(a["out32"].view(torch.int32), b["out32"].view(torch.int32)), f"{what}: fp32 output differs"


@pytest.mark.parametrize("w", FIXTURES, ids=[f.name for f in FIXTURES])
def test_persistent_fixture_matches_oracle_and_per_split_grid(w):
    q, k, v, lens = make_inputs(w)
    per_split = run(w, q, k, v, lens, persistent=0)
    pers = run(w, q, k, v, lens, persistent=ALL)
    assert per_split["plan"].persistent == 0 and pers["plan"].persistent > 0
    assert pers["deverr"] == 0
    check(pers, oracle_ref(w, q, k, v, lens), what=w.name)
    _same_bits(pers, per_split, w.name)


MANY_ITEMS = ["batch16_ragged_llama", "ring_wrap_33000", "tile_pm1_d512", "batch4_mqa_with_empty",
              "batch3_ring_mixed", "mha_d64"]


@pytest.mark.parametrize("blocks", [1, 2, 3, 5])
@pytest.mark.parametrize("name", MANY_ITEMS)
def test_few_persistent_blocks_run_many_items(name, blocks):
    w = next(f for f in FIXTURES if f.name == name)
    q, k, v, lens = make_inputs(w)
    per_split = run(w, q, k, v, lens, persistent=0)
    pers = run(w, q, k, v, lens, persistent=blocks)
    assert pers["plan"].persistent == min(blocks, pers["plan"].num_splits * w.NKV * w.B)
    assert pers["deverr"] == 0
    check(pers, oracle_ref(w, q, k, v, lens), what=f"{name} P={blocks}")
    _same_bits(pers, per_split, f"{name} P={blocks}")


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_persistent_grid_at_any_split_count(splits):
    """S = 1 (each item writes its rows directly, an empty sequence writes
    zeros) through many splits, on three blocks."""
    w = W("pers_splits", 6, 32, 8, 128, 600, 0, lens=(0, 600, 1, 255, 599, 64), seed=81)
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    per_split = run(w, q, k, v, lens, splits=splits, persistent=0)
    pers = run(w, q, k, v, lens, splits=splits, persistent=3)
    assert pers["plan"].num_splits == splits and pers["plan"].persistent == 3
    check(pers, ref, what=f"S={splits}")
    _same_bits(pers, per_split, f"S={splits}")


def test_persistent_workspace_reused_across_calls_and_graph_replay():
    """One workspace for several direct calls and for graph replays: the work
    counter is zero again after each call, so every call sees all items."""
    w = next(f for f in FIXTURES if f.name == "batch16_ragged_llama")
    q, k, v, lens = make_inputs(w)
    want = run(w, q, k, v, lens, persistent=0)
    dev = torch.device("cuda")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), lens.to(dev)
    plan = fd.fd_plan(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window)
    fd.fd_plan_persistent(plan, 1)
    plan.persistent = min(plan.persistent, 4)
    ws = Guarded(plan.workspace_bytes, dev, fill=0xFF)
    ws.body[: plan.workspace_zero_bytes].zero_()
    out = torch.full_like(qd, float("nan"))

    def call(stream=None):
        fd.fd_decode_attn_ex(plan, ws.ptr(), plan.workspace_bytes, None, qd, kd, vd, out, ld, w.B, w.NH, w.NKV,
                             w.HS, w.capacity, w.window, w.scale, stream=stream)

    def counter_zero():
        return bool((ws.body[: plan.workspace_zero_bytes] == 0).all().item())

    for _ in range(3):
        out.fill_(float("nan"))
        call()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(torch.int16), want["out"].view(torch.int16))
        assert counter_zero()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(stream=s)
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(torch.int16), want["out"].view(torch.int16))
        assert counter_zero()
    assert ws.canaries_intact()
    assert fd.fd_get_device_error() == 0


@pytest.mark.parametrize("blocks", [2, ALL])
@pytest.mark.parametrize("name", ["batch16_ragged_llama", "ring_wrap_33000", "tile_pm1_d512", "g16_d64"])
def test_persistent_e4m3_cache(name, blocks):
    w = next(f for f in FIXTURES if f.name == name)
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    per_split = run_fp8(w, q, k8, v8, ks, vs, lens, persistent=0)
    pers = run_fp8(w, q, k8, v8, ks, vs, lens, persistent=blocks)
    assert pers["plan"].persistent > 0 and pers["deverr"] == 0
    check(pers, oracle_ref_fp8(w, q, k8, v8, ks, vs, lens), what=f"{name} P={blocks}")
    _same_bits(pers, per_split, f"{name} P={blocks}")


@pytest.mark.parametrize("name", ["llama_ragged", "gemma_mqa_long"])
def test_persistent_full_size_workloads(name):
    """The two multi-wave workloads at full size: the persistent grid gives the
    per-split grid's bits, and sampled rows match the oracle."""
    w = WORKLOADS[name]
    dev = torch.device("cuda")
    q, k, v, lens = make_inputs(w, device=dev)
    pers = run(w, q, k, v, lens, inputs_on_device=True, persistent=ALL)
    per_split = run(w, q, k, v, lens, inputs_on_device=True, persistent=0)
    assert pers["plan"].persistent > 0 and pers["deverr"] == 0
    assert torch.isfinite(pers["out32"]).all()
    _same_bits(pers, per_split, name)
    rows = _sample_rows(w, lens)
    qh, kh, vh = q.cpu(), k.cpu(), v.cpu()
    del q, k, v
    torch.cuda.empty_cache()
    check(pers, oracle_ref(w, qh, kh, vh, lens, rows=rows), rows=rows, what=name)
