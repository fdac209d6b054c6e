"""Reads before the lengths are known: the plan's min_len bound.

"Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus (Part 2)",
section "One KV head breaks the textbook": the kernel reads only the live band
[max(0, len - window), len), never the allocation. A split block may copy a
tile before its sequence's length arrives only when every length the caller
allows (>= the plan's min_len) makes that tile live. These tests run with
every slot outside the band NaN-poisoned, so a dead slot that reached the
output would show, and check:

  * with the bound kept (min_len <= every len_b), the result equals the
    min_len = 0 result bit for bit and the oracle within tolerance, and no
    error bit is raised;
  * with the bound broken (min_len > some len_b), tiles copied early hold dead
    (NaN) slots, yet the result is still exact, the split counters are back
    at zero, and FD_DEVERR_MIN_LEN is raised;
  * for the bf16 and the E4M3 cache, several split counts, empty sequences.

The DRAM bytes a call reads are measured with ncu (profiles/), not here.
"""

import pytest
import torch

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import Workload as W, make_inputs, make_inputs_fp8
from harness import check, oracle_ref, oracle_ref_fp8, run, run_fp8

pytestmark = pytest.mark.gpu

# (workload, min_len kept, min_len broken)
CASES = [
    (W("tiny_half", 1, 32, 8, 128, 512, 0, lens=(256,), seed=701), 256, 512),
    (W("ring_not_full", 1, 16, 8, 256, 1024, 1024, lens=(700,), seed=702), 700, 1024),
    (W("ring_full", 1, 16, 8, 256, 1024, 1024, lens=(4000,), seed=703), 1024, 9000),
    (W("mqa_short", 1, 16, 1, 512, 4096, 0, lens=(1500,), seed=704), 1500, 4096),
    (W("mqa_two", 2, 16, 1, 512, 4096, 0, lens=(4096, 1234), seed=705), 1234, 4096),
    (W("gqa_d64", 1, 8, 2, 64, 2048, 0, lens=(1000,), seed=706), 1000, 2048),
    (W("empty_seq", 1, 16, 8, 256, 512, 0, lens=(0,), seed=707), 0, 512),
    (W("ragged_lpt", 3, 32, 8, 128, 1024, 0, lens=(1024, 5, 333), seed=708), 5, 1024),
]


@pytest.mark.parametrize("splits", [0, 1, 3, 7])
@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_min_len_kept_equals_no_bound_and_oracle(case, splits):
    w, kept, _ = case
    q, k, v, lens = make_inputs(w)
    base = run(w, q, k, v, lens, splits=splits)
    res = run(w, q, k, v, lens, splits=splits, min_len=kept)
    ref = oracle_ref(w, q, k, v, lens)
    check(res, ref, what=f"{w.name} S={splits} min_len={kept}")
    assert res["deverr"] == 0
    assert torch.equal(res["out32"], base["out32"])
    assert torch.equal(res["out"].view(torch.int16), base["out"].view(torch.int16))


@pytest.mark.parametrize("splits", [0, 1, 3, 7])
@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_min_len_broken_stays_exact_and_is_reported(case, splits):
    w, _, broken = case
    q, k, v, lens = make_inputs(w)
    res = run(w, q, k, v, lens, splits=splits, min_len=broken)
    ref = oracle_ref(w, q, k, v, lens)
    check(res, ref, what=f"{w.name} S={splits} min_len={broken} (broken)")
    assert res["deverr"] & fd.FD_DEVERR_MIN_LEN
    assert res["deverr"] & ~(fd.FD_DEVERR_MIN_LEN | fd.FD_DEVERR_LEN_CLAMPED) == 0


@pytest.mark.parametrize("cluster", [2, 4, 8])
def test_min_len_with_clusters(cluster):
    """Blocks of a cluster read their early tiles too; kept and broken bounds."""
    w = W("ring_cluster", 1, 16, 8, 256, 1024, 1024, lens=(700,), seed=709)
    q, k, v, lens = make_inputs(w)
    ref = oracle_ref(w, q, k, v, lens)
    base = run(w, q, k, v, lens, splits=16, cluster=cluster)
    res = run(w, q, k, v, lens, splits=16, cluster=cluster, min_len=700)
    check(res, ref, what=f"cluster {cluster} min_len kept")
    assert res["deverr"] == 0
    assert torch.equal(res["out32"], base["out32"])
    res = run(w, q, k, v, lens, splits=16, cluster=cluster, min_len=1024)
    check(res, ref, what=f"cluster {cluster} min_len broken")
    assert res["deverr"] & fd.FD_DEVERR_MIN_LEN


FP8_CASES = [c for c in CASES if c[0].name in ("tiny_half", "ring_not_full", "mqa_two", "empty_seq")]


@pytest.mark.parametrize("case", FP8_CASES, ids=[c[0].name for c in FP8_CASES])
def test_min_len_e4m3_kept_and_broken(case):
    w, kept, broken = case
    q, k8, v8, ks, vs, lens = make_inputs_fp8(w)
    ref = oracle_ref_fp8(w, q, k8, v8, ks, vs, lens)
    base = run_fp8(w, q, k8, v8, ks, vs, lens)
    res = run_fp8(w, q, k8, v8, ks, vs, lens, min_len=kept)
    check(res, ref, what=f"{w.name} e4m3 min_len={kept}")
    assert res["deverr"] == 0
    assert torch.equal(res["out32"], base["out32"])
    res = run_fp8(w, q, k8, v8, ks, vs, lens, min_len=broken)
    check(res, ref, what=f"{w.name} e4m3 min_len={broken} (broken)")
    assert res["deverr"] & fd.FD_DEVERR_MIN_LEN


def test_min_len_plan_field_survives_overrides():
    plan = fd.fd_plan(1, 16, 8, 256, 1024, 1024)
    assert plan.min_len == 0
    fd.fd_plan_min_len(plan, 1024)
    fd.fd_plan_override(plan, 5, 0, 0, -1)
    fd.fd_plan_persistent(plan, 0)
    assert plan.min_len == 1024
    with pytest.raises(fd.FdError):
        fd.fd_plan_min_len(plan, -1)
