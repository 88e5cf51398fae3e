"""GPU parity of the scalar-gate variant (A_t = alpha_t I, the gated family
NoteBank Sec. 2 names next to the delta rule) against the fp64 oracle: the
chunked prefill (both schedules, sequence segments), the fp32 token-serial
prefill, and the decode step."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "alpha", "beta")


def oracle_ref(inp, S_in=None, q_scale=1.0):
    return oracle.gated(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")), inp["alpha"].cpu().numpy(),
                        inp["beta"].cpu().numpy(), S_in=None if S_in is None else S_in.double().cpu().numpy(),
                        q_scale=q_scale)


@pytest.mark.parametrize("N", [1, 63, 64, 65, 300, 1000])
def test_gated_bf16_ragged_with_state_and_q_scale(N):
    dev = cuda_device()
    inp = synthetic.gdn_inputs(2, 3, N, dtype=torch.bfloat16, seed=800 + N)
    S_in = torch.randn((2, 3, 128, 128), generator=torch.Generator().manual_seed(N)) * 0.1
    o, S = la.la_gated_prefill(*(inp[n].to(dev) for n in NAMES), S_in=S_in.to(dev), q_scale=0.5)
    torch.cuda.synchronize()
    ref = oracle_ref(inp, S_in=S_in, q_scale=0.5)
    tol = TOL[torch.bfloat16]
    assert rel_err(to_np(o), ref["o"]) < tol
    assert rel_err(to_np(S), ref["S"]) < tol
    assert la.la_device_status() == la.LA_OK


def test_gated_fp32_token_serial():
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 2, 200, dtype=torch.float32, seed=81)
    S_in = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(8)) * 0.1
    o, S = la.la_gated_prefill(*(inp[n].to(dev) for n in NAMES), S_in=S_in.to(dev))
    torch.cuda.synchronize()
    ref = oracle_ref(inp, S_in=S_in)
    assert rel_err(to_np(o), ref["o"]) < TOL[torch.float32]
    assert rel_err(to_np(S), ref["S"]) < TOL[torch.float32]


def test_gated_differs_from_delta_rule():
    """Same inputs through both variants: the results must differ (the kernels
    really switch the erase term off), and each must meet its own oracle."""
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 2, 256, dtype=torch.bfloat16, seed=82)
    x = {n: inp[n].to(dev) for n in NAMES}
    og, _ = la.la_gated_prefill(*(x[n] for n in NAMES))
    od, _ = la.la_gdn_prefill(*(x[n] for n in NAMES))
    torch.cuda.synchronize()
    ref_g = oracle_ref(inp)
    ref_d = oracle.gdn(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")), inp["alpha"].numpy(),
                       inp["beta"].numpy())
    tol = TOL[torch.bfloat16]
    assert rel_err(to_np(og), ref_g["o"]) < tol
    assert rel_err(to_np(od), ref_d["o"]) < tol
    assert rel_err(ref_g["o"], ref_d["o"]) > 3 * tol


@pytest.mark.parametrize("N", [6144, 7990])
def test_gated_segments_and_both_schedules(N):
    """Few heads and a long sequence: sequence segments (the segment maps of
    a scalar gate are pure decays); the one-kernel schedule (minimum
    workspace) must agree with the records schedule and both with the oracle."""
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 2, N, dtype=torch.bfloat16, seed=830 + N)
    g = torch.Generator().manual_seed(N)
    inp["alpha"] = torch.exp(-(0.0005 + 0.0005 * torch.rand(inp["alpha"].shape, generator=g))).contiguous()
    x = {n: inp[n].to(dev) for n in NAMES}
    need_min = la.la_gdn_prefill_workspace_size_min(*(x[n] for n in NAMES))
    assert need_min > 0, "expected the segment path"
    S_in = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(3)) * 0.1
    ref = oracle_ref(inp, S_in=S_in)
    tol = TOL[torch.bfloat16]
    outs = []
    for ws in (None, torch.empty(need_min, dtype=torch.uint8, device=dev)):
        o, S = la.la_gated_prefill(*(x[n] for n in NAMES), S_in=S_in.to(dev), workspace=ws)
        torch.cuda.synchronize()
        assert rel_err(to_np(o), ref["o"]) < tol
        assert rel_err(to_np(S), ref["S"]) < tol
        outs.append((to_np(o), to_np(S)))
    assert rel_err(outs[0][0], outs[1][0]) < 1e-2 and rel_err(outs[0][1], outs[1][1]) < 1e-2
    assert la.la_device_status() == la.LA_OK


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gated_decode_steps_and_prefill_continuation(dtype):
    """Decode steps from a non-zero state, then: prefill of the first part
    followed by decode of the rest equals the oracle over the whole sequence."""
    dev = cuda_device()
    S, H, steps = 4, 3, 20
    g = synthetic.gdn_inputs(S, H, steps, dtype=dtype, seed=84)
    S0 = torch.randn((S, H, 128, 128), generator=torch.Generator().manual_seed(9)) * 0.05
    state = S0.to(dev).contiguous()
    outs = []
    for t in range(steps):
        outs.append(to_np(la.la_decode_step(la.LA_VARIANT_GATED, *(g[n][:, :, t].contiguous().to(dev)
                                                                    for n in ("q", "k", "v")),
                                            state, alpha=g["alpha"][:, :, t].contiguous().to(dev),
                                            beta=g["beta"][:, :, t].contiguous().to(dev))))
    ref = oracle_ref(g, S_in=S0)
    tol = TOL[dtype]
    assert rel_err(np.stack(outs, axis=2), ref["o"]) < tol
    assert rel_err(to_np(state), ref["S"]) < tol
    # prefill 12 tokens, decode the last 8
    first = {n: g[n][:, :, :12].contiguous().to(dev) for n in NAMES}
    o_p, st = la.la_gated_prefill(*(first[n] for n in NAMES), S_in=S0.to(dev))
    dec = []
    for t in range(12, steps):
        dec.append(to_np(la.la_decode_step(la.LA_VARIANT_GATED, *(g[n][:, :, t].contiguous().to(dev)
                                                                   for n in ("q", "k", "v")),
                                           st, alpha=g["alpha"][:, :, t].contiguous().to(dev),
                                           beta=g["beta"][:, :, t].contiguous().to(dev))))
    assert rel_err(to_np(o_p), ref["o"][:, :, :12]) < tol
    assert rel_err(np.stack(dec, axis=2), ref["o"][:, :, 12:]) < tol
    assert rel_err(to_np(st), ref["S"]) < tol


def test_gated_full_size():
    """The benchmark's scalar-gate launch: B=4, H=16, N=16384 bf16 / fp32
    state, run through the scan's scalar-gate order; every head checked
    against the oracle on every token and every state entry."""
    dev = cuda_device()
    w = synthetic.WORKLOADS["gdn_prefill"]
    inp = synthetic.workload_inputs("gdn_prefill", device=dev)
    o, S = la.la_gated_prefill(*(inp[n] for n in NAMES))
    torch.cuda.synchronize()
    assert la.la_device_status() == la.LA_OK
    tol = TOL[torch.bfloat16]
    for b in range(w.B):  # one batch row (16 heads) of oracle work at a time
        sub = {n: inp[n][b:b + 1].cpu() for n in NAMES}
        ref = oracle_ref(sub)
        assert rel_err(to_np(o[b:b + 1]), ref["o"]) < tol, b
        assert rel_err(to_np(S[b:b + 1]), ref["S"]) < tol, b
