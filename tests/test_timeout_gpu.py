"""The give-up path of the tensor-core prefill's bounded waits, exercised without a GPU fault.

Every wait inside the prefill kernel is bounded; one that runs out records GDN_ERR_TIMEOUT in the
device status word, the CTA's roles stop, everything already in flight is drained and the CTA
frees its tensor memory.  The test hook gdn_test_stall_prefill makes every CTA first wait on a
barrier that nothing arrives at (a flag nobody sets), and gdn_set_wait_limit_ns lowers the bound
to 20 microseconds so that this wait runs out quickly.  The test checks that such a call returns,
that the status word reads GDN_ERR_TIMEOUT, and that a normal call afterwards, in the same
process, matches the oracle with a clean status word: the aborted CTAs left no tensor memory
allocated and nothing waiting."""
import pytest
import torch

import gated_delta_rule_20_gb300 as gdn
import workloads
from gated_delta_rule_20_gb300 import _binding as B
from gpu_util import check, oracle_for

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _prefill(x):
    st = x["state"].clone()
    out, st = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st, single_pass=True)
    torch.cuda.synchronize()
    return out, st


@pytest.mark.parametrize("seqs", [1, 4])
def test_prefill_wait_timeout_reports_and_recovers(seqs):
    # bf16, Dk = Dv = 128 (the tensor-core path), `seqs` CTAs of four chunks each
    w = workloads.PREFILL.with_(B=1, Hk=1, Hv=seqs, S=256, seed=61 + seqs)
    x = workloads.make_inputs(w, device=DEV)
    gdn.device_status(0, clear=True)
    try:
        B.set_wait_limit_ns(0, 20000)  # 20 us
        B.test_stall_prefill(0, True)
        _prefill(x)                    # returns: no wait is left spinning
        code = gdn.device_status(0, clear=True)
    finally:
        B.test_stall_prefill(0, False)
        B.set_wait_limit_ns(0, 0)      # the default second again
    assert code == gdn.GDN_ERR_TIMEOUT
    # the same process, the default limit: correct results and a clean status word
    out, st = _prefill(x)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "prefill after an aborted call")
    assert gdn.device_status(0, clear=True) == 0
