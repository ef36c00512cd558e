"""Failure detection without a GPU fault: the test hook makes the attention
kernel's producer withhold one K/V copy, so the consumer's bounded wait
(limited to 20 ms here) expires.  The kernel records ULY_ERR_TIMEOUT, drains,
frees TMEM and returns; the context stays usable and the next call is
correct."""
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fill", [0, 1, 5])
def test_withheld_copy_times_out_and_recovers(fill):
    import torch
    from ulysses_sequence_attention_uly_gb300 import ULY_ERR_TIMEOUT
    w = synth.WORKLOADS["tiny"].scaled(S_l=300, R=16, valid=None)
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    good = H.run_fused(plan, w, d)
    assert plan.sync_status() == 0
    plan.set_wait_limit(20_000_000)
    plan.test_withhold_fill(fill)
    H.run_fused(plan, w, d)
    assert plan.sync_status() == ULY_ERR_TIMEOUT
    # the status word was cleared and the context still works
    plan.test_withhold_fill(-1)
    again = H.run_fused(plan, w, d)
    assert plan.sync_status() == 0
    torch.cuda.synchronize()
    for a, b in zip(good, again):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
