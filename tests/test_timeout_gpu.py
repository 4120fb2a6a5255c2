"""A bounded on-chip wait that runs out, on the GPU, without a fault.

The testing aid gdn_testing_wait_limit shortens every hand-off wait of the prefill
kernel and makes the chunk-local group of each CTA withhold its first "operands
ready" hand-off, so the wait for it gives up by design.  The call must return, the
device error word must report GDN_DEVERR_TIMEOUT, and a normal call right after, on
the same context, must still match the oracle ("flashinfer.gdn_prefill": invalid
inputs fail closed; every wait of the kernel is bounded and drains before the CTA
exits).
"""
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _restore_limits():
    from gated_delta_rule_24_gb300 import build
    build.build()
    gdn.gdn_init(0)
    assert gdn.device_status() == 0
    yield
    gdn.testing_wait_limit(0, False)
    gdn.testing_force_splits(0)


def _run(p):
    out, st = gdn.run_problem(p, device=DEV)
    torch.cuda.synchronize()  # the call has returned and its kernels have ended
    return out, st


@pytest.mark.parametrize("splits", [0, 3])
def test_wait_that_runs_out_reports_timeout_and_leaves_the_context_usable(splits):
    p = W.make_problem([300, 64, 0, 650, 130], 2, 4, gates="mamba", init="fp32", init_std=0.05, seed=81,
                       batch_invariant=splits == 0)
    gdn.testing_force_splits(splits)
    gdn.testing_wait_limit(50_000, True)  # 50 us; the first hand-off of every CTA withheld
    _run(p)
    word = gdn.device_status()
    assert word & gdn.binding.DEVERR_TIMEOUT, word
    gdn.testing_wait_limit(0, False)
    out, st = _run(p)
    assert gdn.device_status() == 0
    compare(p, out, st)


def test_testing_aids_validate_their_arguments():
    with pytest.raises(gdn.GdnError):
        gdn.testing_wait_limit(10, False)
    with pytest.raises(gdn.GdnError):
        gdn.testing_force_splits(9)
