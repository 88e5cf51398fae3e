"""GPU parity of BASED with a fixed per-head decay (BASED notes, the decay
paragraph after Table 7; s_i = lambda_h s_{i-1} + phi(k_i) v_i^T, z likewise)
against the fp64 oracle: the chunked bf16 prefill, the token-serial fp32
prefill and the decode step, with ragged lengths, an incoming state, the
end values lambda = 1 and lambda = 0, and prefill followed by decode."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu

# one head per regime: long memory, short memory, no decay, a reset every token
DECAYS = [0.995, 0.9, 1.0, 0.0, 0.5, 0.97]


def run(inp, dev, lam, s_in=None, z_in=None, eps=0.0):
    H = inp["q"].shape[1]
    decay = torch.tensor(lam[:H], dtype=torch.float32)
    y, s, z = la.la_based_prefill(*(inp[n].to(dev) for n in ("q", "k", "v")),
                                  s_in=None if s_in is None else s_in.to(dev),
                                  z_in=None if z_in is None else z_in.to(dev), eps=eps, decay=decay.to(dev))
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")),
                        s_in=None if s_in is None else s_in.double().numpy(),
                        z_in=None if z_in is None else z_in.double().numpy(), eps=eps,
                        decay=decay.double().numpy())
    torch.cuda.synchronize()
    return (to_np(y), to_np(s), to_np(z)), ref


def check(got, ref, tol):
    for name, x in zip(("y", "s", "z"), got):
        err = rel_err(x, ref[name])
        assert err < tol, f"{name}: {err:.3e}"


@pytest.mark.parametrize("N", [1, 100, 127, 128, 129, 300, 1000])
def test_decay_bf16_chunked_ragged_with_state(N):
    dev = cuda_device()
    inp = synthetic.taylor_inputs(2, 6, N, dtype=torch.bfloat16, seed=900 + N)
    g = torch.Generator().manual_seed(N)
    s_in = torch.randn((2, 6, la.TAYLOR_D, 64), generator=g) * 0.1
    z_in = torch.rand((2, 6, la.TAYLOR_D), generator=g) + 0.5
    got, ref = run(inp, dev, DECAYS, s_in=s_in, z_in=z_in, eps=1e-3)
    check(got, ref, TOL[torch.bfloat16])
    assert la.la_device_status() == la.LA_OK


def test_decay_one_matches_undecayed_kernel_exactly():
    """lambda = 1 takes the decay instantiation of the kernel, whose factors
    are then all exactly one, and whose fp32-path features round to the same
    bf16 as the paired bf16 products: the outputs equal the undecayed
    instantiation bit for bit."""
    dev = cuda_device()
    inp = synthetic.taylor_inputs(1, 4, 700, dtype=torch.bfloat16, seed=77)
    x = {n: inp[n].to(dev) for n in ("q", "k", "v")}
    y0, s0, z0 = la.la_based_prefill(x["q"], x["k"], x["v"])
    y1, s1, z1 = la.la_based_prefill(x["q"], x["k"], x["v"], decay=torch.ones(4, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(y1, y0) and torch.equal(s1, s0) and torch.equal(z1, z0)


def test_decay_fp32_token_serial():
    dev = cuda_device()
    inp = synthetic.taylor_inputs(1, 6, 200, dtype=torch.float32, seed=91)
    g = torch.Generator().manual_seed(9)
    s_in = torch.randn((1, 6, la.TAYLOR_D, 64), generator=g) * 0.1
    z_in = torch.rand((1, 6, la.TAYLOR_D), generator=g) + 0.5
    got, ref = run(inp, dev, DECAYS, s_in=s_in, z_in=z_in)
    check(got, ref, TOL[torch.float32])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decay_decode_and_prefill_continuation(dtype):
    """Prefill of the first 150 tokens (the chunked kernel for bf16) then
    decode steps for the rest equal the oracle over the whole sequence."""
    dev = cuda_device()
    S, H, N, first = 3, 6, 170, 150
    inp = synthetic.taylor_inputs(S, H, N, dtype=dtype, seed=93)
    decay = torch.tensor(DECAYS, dtype=torch.float32)
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")), decay=decay.double().numpy())
    x = {n: inp[n].to(dev) for n in ("q", "k", "v")}
    y, s, z = la.la_based_prefill(*(x[n][:, :, :first].contiguous() for n in ("q", "k", "v")), decay=decay.to(dev))
    outs = []
    for t in range(first, N):
        outs.append(to_np(la.la_decode_step(la.LA_VARIANT_TAYLOR, *(x[n][:, :, t].contiguous() for n in ("q", "k", "v")),
                                            s, z=z, decay=decay.to(dev))))
    torch.cuda.synchronize()
    tol = TOL[dtype]
    assert rel_err(to_np(y), ref["y"][:, :, :first]) < tol
    assert rel_err(np.stack(outs, axis=2), ref["y"][:, :, first:]) < tol
    assert rel_err(to_np(s), ref["s"]) < tol and rel_err(to_np(z), ref["z"]) < tol


def test_decay_zero_head_returns_current_value():
    """lambda = 0 keeps only the current token: y_i = v_i (BASED map, eps = 0)."""
    dev = cuda_device()
    inp = synthetic.taylor_inputs(1, 2, 260, dtype=torch.bfloat16, seed=95)
    y, _, _ = la.la_based_prefill(*(inp[n].to(dev) for n in ("q", "k", "v")),
                                  decay=torch.zeros(2, device=dev))
    torch.cuda.synchronize()
    assert rel_err(to_np(y), inp["v"].float().numpy()) < TOL[torch.bfloat16]


def test_decay_full_size():
    """The benchmark's launch: B=8, H=16, N=4096 bf16 with lambda_h = 1 - 2^-(5 + h mod 8), a spread from
    a 32- to a 4096-token memory; every output and final state against the oracle."""
    dev = cuda_device()
    inp = synthetic.workload_inputs("based_prefill", device=dev)
    H = inp["q"].shape[1]
    lam = [1.0 - 2.0 ** -(5 + h % 8) for h in range(H)]
    got, ref = run(inp, dev, lam)
    check(got, ref, TOL[torch.bfloat16])
    assert la.la_device_status() == la.LA_OK
