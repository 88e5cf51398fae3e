"""Decode steps launched back to back on one stream.

Each decode kernel is launched as a programmatic dependent: it may be
scheduled while the step before it still runs and waits for that step only
before its first memory access.  Steps launched back to back must therefore
give exactly the bits of the same steps with a device synchronisation between
them (same kernels, same inputs, same order)."""
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import synthetic
from tests.helpers import cuda_device

pytestmark = pytest.mark.gpu

S, H, STEPS = 64, 8, 24


def _run(variant, inputs, sync):
    dev = cuda_device()
    if variant == "gdn":
        state = torch.zeros((S, H, 128, 128), device=dev)
        z = None
    else:
        state = torch.zeros((S, H, la.TAYLOR_D, 64), device=dev)
        z = torch.zeros((S, H, la.TAYLOR_D), device=dev)
    outs = []
    for x in inputs:
        out = torch.empty((S, H, 128 if variant == "gdn" else 64), dtype=torch.bfloat16, device=dev)
        if variant == "gdn":
            la.la_decode_step(la.LA_VARIANT_GDN, x["q"], x["k"], x["v"], state, alpha=x["alpha"], beta=x["beta"],
                              out=out)
        else:
            la.la_decode_step(la.LA_VARIANT_TAYLOR, x["q"], x["k"], x["v"], state, z=z, out=out)
        outs.append(out)
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return outs, state, z


@pytest.mark.parametrize("variant", ["gdn", "taylor"])
def test_back_to_back_decode_steps_match_synchronised_steps(variant):
    dev = cuda_device()
    inputs = [synthetic.decode_step_inputs(S, H, t, seed=5, device=dev)[variant] for t in range(STEPS)]
    torch.cuda.synchronize()
    a_out, a_state, a_z = _run(variant, inputs, sync=False)
    b_out, b_state, b_z = _run(variant, inputs, sync=True)
    for t in range(STEPS):
        assert torch.equal(a_out[t], b_out[t]), f"output of step {t}"
    assert torch.equal(a_state, b_state)
    if a_z is not None:
        assert torch.equal(a_z, b_z)
    assert la.la_device_status() == la.LA_OK


@pytest.mark.parametrize("d", [64, 32])
def test_back_to_back_window_steps_match_synchronised_steps(d):
    """d = 64 takes the staged kernel, d = 32 the direct one; the ring wraps twice."""
    dev = cuda_device()
    window = 16
    g = torch.Generator().manual_seed(d)
    xs = [tuple(torch.randn((S, H, d), generator=g).to(torch.bfloat16).to(dev) for _ in range(3))
          for _ in range(2 * window + 3)]
    kc0 = torch.randn((S, H, window, d), generator=g).to(torch.bfloat16).to(dev)
    vc0 = torch.randn((S, H, window, d), generator=g).to(torch.bfloat16).to(dev)
    start = torch.arange(S, dtype=torch.int64) % (2 * window)  # some rings still filling, some full
    pos = [(start + t).to(dev) for t in range(len(xs))]  # on the device first: nothing between the steps

    def run(sync):
        kc, vc = kc0.clone(), vc0.clone()
        outs = []
        for t, (q, k, v) in enumerate(xs):
            outs.append(la.la_swa_decode_step(q, k, v, kc, vc, pos[t]))
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return outs, kc, vc

    a_out, a_kc, a_vc = run(False)
    b_out, b_kc, b_vc = run(True)
    for t in range(len(xs)):
        assert torch.equal(a_out[t], b_out[t]), f"output of step {t}"
    assert torch.equal(a_kc, b_kc) and torch.equal(a_vc, b_vc)
    assert la.la_device_status() == la.LA_OK
