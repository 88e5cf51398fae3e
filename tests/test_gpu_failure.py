"""The bounded-wait error path: a wait that runs out sets the device status
word (LA_ERR_TIMEOUT on the host) instead of hanging, and the context stays
usable.  The wait runs out because nothing arrives on its barrier; no fault,
trap or unbounded wait is involved."""
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    dev = cuda_device()
    assert la.la_device_status(clear=True) == la.LA_OK
    # nothing arrives: the wait gives up after 50 ms
    assert la.la_selftest_bounded_wait(False, 50_000_000) == la.LA_OK
    assert la.la_device_status(clear=False) == la.LA_ERR_TIMEOUT
    assert la.la_device_status(clear=True) == la.LA_ERR_TIMEOUT   # read and clear
    assert la.la_device_status(clear=True) == la.LA_OK
    # the thread arrives itself: no timeout
    assert la.la_selftest_bounded_wait(True, 50_000_000) == la.LA_OK
    assert la.la_device_status(clear=True) == la.LA_OK
    # limits outside [1 ms, 2 s] are rejected before any launch
    assert la.la_selftest_bounded_wait(False, 10) == la.LA_ERR_INVALID_ARGUMENT
    assert la.la_selftest_bounded_wait(False, 5_000_000_000) == la.LA_ERR_INVALID_ARGUMENT
    # the context is still usable: a tensor-core prefill runs and is correct
    g = synthetic.gdn_inputs(1, 2, 100, dtype=torch.bfloat16, seed=51)
    o, S = la.la_gdn_prefill(*(g[n].to(dev) for n in ("q", "k", "v", "alpha", "beta")))
    torch.cuda.synchronize()
    ref = oracle.gdn(*(synthetic.to_oracle(g[n]) for n in ("q", "k", "v")), g["alpha"].numpy(), g["beta"].numpy())
    assert rel_err(to_np(o), ref["o"]) < TOL[torch.bfloat16]
    assert la.la_device_status(clear=True) == la.LA_OK
