"""The bounded-wait path of the persistent tcgen05 kernel, made to run out
on purpose in its allowed form: a short wait limit (1 ms) and a host-side
test hook that makes the first CTA's TMA producer take one pipeline stage
without issuing its copies.  The MMA warp's wait for that stage then ends
by its limit, not by an arrival: the kernel must record the timeout in the
handle's device status word, wait for its own copies and MMAs in flight,
free its TMEM and return.  Nothing faults, traps or hangs; the context stays
usable, so the next call on the same handle must be correct again.
"""
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
from tests import _cases

pytestmark = pytest.mark.gpu

DEVICE_TIMEOUT = 6


@pytest.fixture()
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


@pytest.mark.parametrize("mode,transA,skip", [("bf16", False, 3), ("bf16", False, 1), ("tf32", False, 9),
                                               ("tf32", True, 3)])
def test_wait_runs_out_then_next_call_is_correct(h, mode, transA, skip):
    M, N, K = 300, 264, 1024  # 3 x 3 tiles of 128 columns, 16-32 K blocks per tile
    ops, _ = _cases.make(mode, M, N, K, transA, False, seed=311, dist="normal")
    h.set_option("family", "tc")
    h.set_option("tile_n", 128)
    h.set_option("split_k", 1)  # CTA 0 takes one whole tile: 16 (BF16) or 32 (TF32) stages
    h.set_option("wait_limit_us", 1000)
    h.set_option("fault_skip_stage", skip)
    C = torch.zeros((M, N), device="cuda")
    h.run(ops.A, ops.B, C, mode=mode, transA=transA)
    assert h.check_device() == DEVICE_TIMEOUT
    plan = h.plan()
    assert plan["family"] == "tc" and plan["cluster"] == 1 and plan["tile_n"] == 128 and plan["split_k"] == 1, plan
    # the status word was cleared by the check; the GPU answers and the next
    # call on the same handle (hook off, default limit) is right again
    assert h.check_device() == 0
    h.set_option("fault_skip_stage", 0)
    h.set_option("wait_limit_us", 0)
    _cases.run_and_check(h, mode, M, N, K, transA, False, seed=312, dist="normal")
    _cases.run_and_check(h, mode, M, N, K, transA, False, seed=313, dist="int", exact=True)


def test_short_limit_alone_changes_nothing(h):
    """A 1 ms limit on a call whose stages all arrive: no timeout, exact result."""
    h.set_option("wait_limit_us", 1000)
    _cases.run_and_check(h, "bf16", 1000, 1000, 2048, seed=314, dist="int", exact=True)
    assert h.check_device() == 0
