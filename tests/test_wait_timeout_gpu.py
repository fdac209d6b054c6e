"""The bounded waits give up, report, and leave the GPU usable.

Every pipeline wait of the kernels is bounded: after a wall-time limit it
raises FD_DEVERR_WAIT_TIMEOUT in the device error word and returns, and the
kernel runs to its end, so no wait can hang the GPU. These tests make such a
wait run out on purpose, without faulting anything: through the library's
test hook (fd_debug_withhold_copies) the split blocks never issue the copies
of one of their tiles - nothing is left in flight - so the consumers' wait for
that tile has nothing to wait for. The limit is shortened to 100 us. Then:

  * the call returns and the stream completes;
  * fd_get_device_error reports FD_DEVERR_WAIT_TIMEOUT;
  * no output buffer's guard canaries were touched;
  * with the hook off, the next call on the same device is exact against the
    FP64 oracle and raises no error bit.
"""

import pytest

import decode_attention_04_gb300 as fd
from decode_attention_04_gb300.inputs import Workload as W, make_inputs
from harness import check, oracle_ref, run

pytestmark = pytest.mark.gpu

LIMIT_NS = 100_000

CASES = [
    # (workload, splits (0: the plan's), tile of each split whose copies are withheld)
    (W("ring_first_tile", 1, 16, 8, 256, 1024, 1024, lens=(5000,), seed=801), 0, 0),
    (W("mqa_third_tile", 1, 16, 1, 512, 8192, 0, lens=(8192,), seed=802), 4, 2),
    (W("llama_second_tile", 2, 32, 8, 128, 4096, 0, lens=(4096, 3000), seed=803), 2, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0].name for c in CASES])
def test_withheld_tile_times_out_reports_and_next_call_is_exact(case):
    w, splits, tile = case
    q, k, v, lens = make_inputs(w)
    fd.fd_debug_withhold_copies(tile, LIMIT_NS)
    try:
        bad = run(w, q, k, v, lens, splits=splits)
    finally:
        fd.fd_debug_withhold_copies(-1, 0)
    assert bad["deverr"] & fd.FD_DEVERR_WAIT_TIMEOUT, "the wait for the withheld tile did not give up"
    assert bad["canaries"], "a guard canary was overwritten"
    good = run(w, q, k, v, lens, splits=splits)
    assert good["deverr"] == 0
    check(good, oracle_ref(w, q, k, v, lens), what=f"{w.name} after a timeout")


def test_hook_off_by_default_and_after_reset():
    w, splits, _ = CASES[0]
    q, k, v, lens = make_inputs(w)
    fd.fd_debug_withhold_copies(-1, 0)
    res = run(w, q, k, v, lens, splits=splits)
    assert res["deverr"] == 0
    check(res, oracle_ref(w, q, k, v, lens), what="hook off")
