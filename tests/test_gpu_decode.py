"""GPU parity of the one-token decode steps against the fp64 oracle."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu


def seq_slice(x, t):
    return x[:, :, t].contiguous()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gdn_decode_steps_from_nonzero_state(dtype):
    dev = cuda_device()
    S, H, steps = 5, 3, 24
    g = synthetic.gdn_inputs(S, H, steps, dtype=dtype, seed=21)
    S0 = torch.randn((S, H, 128, 128), generator=torch.Generator().manual_seed(5)) * 0.05
    state = S0.to(dev).contiguous()
    outs = []
    for t in range(steps):
        outs.append(to_np(la.la_decode_step(la.LA_VARIANT_GDN, *(seq_slice(g[n], t).to(dev) for n in ("q", "k", "v")),
                                            state, alpha=g["alpha"][:, :, t].contiguous().to(dev),
                                            beta=g["beta"][:, :, t].contiguous().to(dev))))
    ref = oracle.gdn(*(synthetic.to_oracle(g[n]) for n in ("q", "k", "v")), g["alpha"].numpy(), g["beta"].numpy(),
                     S_in=S0.double().numpy())
    tol = TOL[dtype]
    assert rel_err(np.stack(outs, axis=2), ref["o"]) < tol
    assert rel_err(to_np(state), ref["S"]) < tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_taylor_decode_steps_from_nonzero_state(dtype):
    dev = cuda_device()
    S, H, steps = 4, 3, 24
    t_in = synthetic.taylor_inputs(S, H, steps, dtype=dtype, seed=22)
    gen = torch.Generator().manual_seed(6)
    s0 = torch.randn((S, H, la.TAYLOR_D, 64), generator=gen)
    z0 = torch.rand((S, H, la.TAYLOR_D), generator=gen) + 1.0
    s, z = s0.to(dev).contiguous(), z0.to(dev).contiguous()
    outs = []
    for t in range(steps):
        outs.append(to_np(la.la_decode_step(la.LA_VARIANT_TAYLOR, *(seq_slice(t_in[n], t).to(dev)
                                                                    for n in ("q", "k", "v")), s, z=z, eps=1e-3)))
    ref = oracle.taylor(*(synthetic.to_oracle(t_in[n]) for n in ("q", "k", "v")), s_in=s0.double().numpy(),
                        z_in=z0.double().numpy(), eps=1e-3)
    tol = TOL[dtype]
    assert rel_err(np.stack(outs, axis=2), ref["y"]) < tol
    assert rel_err(to_np(s), ref["s"]) < tol
    assert rel_err(to_np(z), ref["z"]) < tol


def test_decode_fp32_output_and_inplace_alias():
    dev = cuda_device()
    g = synthetic.gdn_inputs(2, 2, 1, seed=23)
    state = torch.zeros((2, 2, 128, 128), device=dev)
    out = la.la_decode_step(la.LA_VARIANT_GDN, *(g[n][:, :, 0].contiguous().to(dev) for n in ("q", "k", "v")),
                            state, alpha=g["alpha"][:, :, 0].contiguous().to(dev),
                            beta=g["beta"][:, :, 0].contiguous().to(dev), out_dtype=torch.float32)
    assert out.dtype == torch.float32
    ref = oracle.gdn(*(synthetic.to_oracle(g[n]) for n in ("q", "k", "v")), g["alpha"].numpy(), g["beta"].numpy())
    assert rel_err(to_np(out), ref["o"][:, :, 0]) < 2e-2


SAMPLE_STEPS = (1, 10, 100, 1000)


def _sample_pairs(S, H, n, seed):
    rng = np.random.default_rng(seed)
    flat = rng.choice(S * H, n, replace=False)
    return [(int(f // H), int(f % H)) for f in sorted(flat)]


@pytest.mark.parametrize("variant", ["gdn", "taylor"])
def test_decode_full_size_1000_steps(variant):
    """256 sequences x 16 heads, 1000 steps from a zero state, the launch the
    benchmark times; outputs and states checked at steps 1, 10, 100, 1000 on a
    sample of (sequence, head) pairs recomputed by the oracle."""
    dev = cuda_device()
    w = synthetic.WORKLOADS["decode"]
    S, H, steps = w.B, w.H, w.N
    pairs = _sample_pairs(S, H, 24, seed=99)
    si = torch.tensor([p[0] for p in pairs], device=dev)
    hi = torch.tensor([p[1] for p in pairs], device=dev)
    if variant == "gdn":
        state = torch.zeros((S, H, 128, 128), device=dev)
        z = None
    else:
        state = torch.zeros((S, H, la.TAYLOR_D, 64), device=dev)
        z = torch.zeros((S, H, la.TAYLOR_D), device=dev)
    hist = {n: [] for n in ("q", "k", "v", "alpha", "beta")}
    got_out, got_state, got_z = {}, {}, {}
    for t in range(steps):
        x = synthetic.decode_step_inputs(S, H, t, seed=w.seed, device=dev)[variant]
        for n in hist:
            if n in x:
                hist[n].append(x[n][si, hi].cpu())
        if variant == "gdn":
            out = la.la_decode_step(la.LA_VARIANT_GDN, x["q"], x["k"], x["v"], state, alpha=x["alpha"], beta=x["beta"])
        else:
            out = la.la_decode_step(la.LA_VARIANT_TAYLOR, x["q"], x["k"], x["v"], state, z=z)
        if t + 1 in SAMPLE_STEPS:
            got_out[t + 1] = to_np(out[si, hi])
            got_state[t + 1] = to_np(state[si, hi])
            if z is not None:
                got_z[t + 1] = to_np(z[si, hi])
    # [P, steps, d] -> oracle layout [P, 1, steps, d]
    seqs = {n: torch.stack(v, dim=1).unsqueeze(1) for n, v in hist.items() if v}
    tol = TOL[torch.bfloat16]
    for n_steps in SAMPLE_STEPS:
        cut = {n: x[:, :, :n_steps].contiguous() for n, x in seqs.items()}
        if variant == "gdn":
            ref = oracle.gdn(*(synthetic.to_oracle(cut[n]) for n in ("q", "k", "v")), cut["alpha"].numpy(),
                             cut["beta"].numpy(), t_samples=[n_steps - 1])
            assert rel_err(got_out[n_steps], ref["o"][:, 0, 0]) < tol, f"output at step {n_steps}"
            assert rel_err(got_state[n_steps], ref["S"][:, 0]) < tol, f"state at step {n_steps}"
        else:
            ref = oracle.taylor(*(synthetic.to_oracle(cut[n]) for n in ("q", "k", "v")), t_samples=[n_steps - 1])
            assert rel_err(got_out[n_steps], ref["y"][:, 0, 0]) < tol, f"output at step {n_steps}"
            assert rel_err(got_state[n_steps], ref["s"][:, 0]) < tol, f"state at step {n_steps}"
            assert rel_err(got_z[n_steps], ref["z"][:, 0]) < tol, f"normaliser at step {n_steps}"
    assert la.la_device_status() == la.LA_OK
