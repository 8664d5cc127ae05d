"""A pipeline wait that runs out, on the GPU, without a fault: with the library's wait limit set to one
microsecond, the GEMMs of a backward whose weight-gradient contractions run over 8192 rows of one
expert (tens of microseconds per output tile) give up waiting, report MOE_STATUS_TIMEOUT in the
status word, drain the copies and tensor-core work they have in flight and return.  The context stays
usable: with the default limit back, the same call gives results bit-identical to a run made before,
within the parity bar of the oracle."""
import pytest
import torch

from helpers import MXFP8_TOL, compare_outputs, oracle_bwd, run_gpu
from moe_expert_layer_routing_gb300.inputs import AFFINITY_ON_I, PREC_MXFP8, make_moe_inputs, small_moe, with_ids

pytestmark = pytest.mark.gpu


def _inputs():
    T, K, E = 8192, 1, 2
    cfg = small_moe("wait_limit", T=T, H=1024, I=256, E=E, K=K, B=128, seed=61, precision=PREC_MXFP8,
                    affinity=AFFINITY_ON_I)
    ids = torch.zeros(T, K, dtype=torch.int32)
    ids[0, 0] = 1   # expert 1 gets one row, expert 0 all the others
    return with_ids(make_moe_inputs(cfg), ids)


def test_short_wait_limit_reports_timeout_and_the_context_stays_usable(set_option):
    import moe_expert_layer_routing_gb300 as mb
    inp = _inputs()
    _, first = run_gpu(inp)
    assert int(first["status"].item()) == 0
    first = {k: v.clone() for k, v in first.items() if v is not None}

    set_option("WAIT_LIMIT_NS", 1000)
    launches = mb.kernel_launches()
    _, timed = run_gpu(inp)          # returns: the host call succeeds, the device reports
    status = int(timed["status"].item())
    assert status & mb.STATUS_TIMEOUT, f"status {status}: no wait ran out"
    assert mb.kernel_launches() > launches

    set_option("WAIT_LIMIT_NS", None)
    assert mb.get_option("WAIT_LIMIT_NS") == 2_000_000_000
    _, again = run_gpu(inp)
    assert int(again["status"].item()) == 0
    for n in ("dx", "dW1", "dW2", "ds"):
        assert torch.equal(again[n], first[n]), n
    compare_outputs(again, oracle_bwd(inp), MXFP8_TOL)
