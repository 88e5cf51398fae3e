"""GPU parity of the Taylor (BASED) prefill against the fp64 oracle."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu


def run_pair(inp, dev, s_in=None, z_in=None, eps=0.0, out_dtype=None):
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    y, s, z = la.la_based_prefill(q, k, v, s_in=None if s_in is None else s_in.to(dev),
                                  z_in=None if z_in is None else z_in.to(dev), eps=eps, out_dtype=out_dtype)
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")),
                        s_in=None if s_in is None else s_in.double().numpy(),
                        z_in=None if z_in is None else z_in.double().numpy(), eps=eps)
    torch.cuda.synchronize()
    return (to_np(y), to_np(s), to_np(z)), ref


def assert_close(got, ref, tol):
    y, s, z = got
    assert rel_err(y, ref["y"]) < tol, f"y: {rel_err(y, ref['y']):.3e}"
    assert rel_err(s, ref["s"]) < tol, f"s: {rel_err(s, ref['s']):.3e}"
    assert rel_err(z, ref["z"]) < tol, f"z: {rel_err(z, ref['z']):.3e}"


def test_taylor_fp32_small_config():
    """Additive Taylor linear attention, fp32: B=1, H=2, N=256, seed 0; 1e-4."""
    dev = cuda_device()
    inp = synthetic.workload_inputs("taylor_fp32_small")
    got, ref = run_pair(inp, dev)
    assert_close(got, ref, TOL[torch.float32])


@pytest.mark.parametrize("N", [1, 15, 63, 64, 65, 127, 128, 129, 257, 1000])
def test_taylor_bf16_ragged_lengths(N):
    dev = cuda_device()
    inp = synthetic.taylor_inputs(2, 3, N, dtype=torch.bfloat16, seed=100 + N)
    got, ref = run_pair(inp, dev)
    assert_close(got, ref, TOL[torch.bfloat16])


def test_taylor_fp32_ragged_with_state_in_and_eps():
    dev = cuda_device()
    inp = synthetic.taylor_inputs(1, 2, 300, dtype=torch.float32, seed=31)
    gen = torch.Generator().manual_seed(3)
    s_in = torch.randn((1, 2, la.TAYLOR_D, 64), generator=gen)
    z_in = torch.rand((1, 2, la.TAYLOR_D), generator=gen) * 3 + 1
    got, ref = run_pair(inp, dev, s_in=s_in, z_in=z_in, eps=0.25)
    assert_close(got, ref, TOL[torch.float32])


def test_taylor_strided_views_and_fp32_output():
    """q, k, v carved out of one interleaved [B, N, H, 96] buffer; y written
    into a [B, N, H, 64] buffer viewed as [B, H, N, 64]."""
    dev = cuda_device()
    B, H, N = 2, 4, 190
    inp = synthetic.taylor_inputs(B, H, N, dtype=torch.bfloat16, seed=32)
    packed = torch.cat([inp["q"], inp["k"], inp["v"]], dim=-1).permute(0, 2, 1, 3).contiguous().to(dev)
    qv = packed[..., :16].permute(0, 2, 1, 3)
    kv = packed[..., 16:32].permute(0, 2, 1, 3)
    vv = packed[..., 32:].permute(0, 2, 1, 3)
    ybuf = torch.empty((B, N, H, 64), dtype=torch.float32, device=dev)
    y = ybuf.permute(0, 2, 1, 3)
    la.la_based_prefill(qv, kv, vv, y=y)
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")))
    torch.cuda.synchronize()
    assert rel_err(to_np(y), ref["y"]) < TOL[torch.bfloat16]


def test_taylor_split_resume_equals_whole():
    dev = cuda_device()
    inp = synthetic.taylor_inputs(2, 2, 333, dtype=torch.bfloat16, seed=33)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    y, s, z = la.la_based_prefill(q, k, v, out_dtype=torch.float32)
    y1, s1, z1 = la.la_based_prefill(q[:, :, :130], k[:, :, :130], v[:, :, :130], out_dtype=torch.float32)
    y2, s2, z2 = la.la_based_prefill(q[:, :, 130:], k[:, :, 130:], v[:, :, 130:], s_in=s1, z_in=z1,
                                     out_dtype=torch.float32)
    # the split moves chunk boundaries (bf16 operand rounding differs): both runs
    # meet the bf16 contract against the oracle and agree to well inside it
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")))
    y12 = to_np(torch.cat([y1, y2], dim=2))
    assert rel_err(y12, ref["y"]) < TOL[torch.bfloat16]
    assert rel_err(to_np(s2), ref["s"]) < TOL[torch.bfloat16] and rel_err(to_np(z2), ref["z"]) < TOL[torch.bfloat16]
    assert rel_err(y12, to_np(y)) < 1e-2
    assert rel_err(to_np(s2), to_np(s)) < 1e-2 and rel_err(to_np(z2), to_np(z)) < 1e-2


def test_taylor_prefill_then_decode_matches_longer_prefill():
    dev = cuda_device()
    inp = synthetic.taylor_inputs(2, 2, 201, dtype=torch.bfloat16, seed=34)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    _, s, z = la.la_based_prefill(q[:, :, :200], k[:, :, :200], v[:, :, :200])
    y_dec = la.la_decode_step(la.LA_VARIANT_TAYLOR, q[:, :, 200].contiguous(), k[:, :, 200].contiguous(),
                              v[:, :, 200].contiguous(), s, z=z)
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")), t_samples=[200])
    assert rel_err(to_np(y_dec), ref["y"][:, :, 0]) < TOL[torch.bfloat16]
    assert rel_err(to_np(s), ref["s"]) < TOL[torch.bfloat16]


def test_taylor_empty_sequence_passes_state():
    dev = cuda_device()
    q = torch.zeros((1, 2, 0, 16), dtype=torch.bfloat16, device=dev)
    v = torch.zeros((1, 2, 0, 64), dtype=torch.bfloat16, device=dev)
    s_in = torch.randn((1, 2, la.TAYLOR_D, 64), device=dev)
    z_in = torch.randn((1, 2, la.TAYLOR_D), device=dev)
    _, s, z = la.la_based_prefill(q, q, v, s_in=s_in, z_in=z_in)
    assert torch.equal(s, s_in) and torch.equal(z, z_in)
    _, s, z = la.la_based_prefill(q, q, v)
    assert torch.count_nonzero(s) == 0 and torch.count_nonzero(z) == 0


def test_based_prefill_full_size():
    """BASED Taylor prefill, bf16 in / fp32 state: B=8, H=16, N=4096, the launch
    the benchmark times; every output and final state against the oracle."""
    dev = cuda_device()
    inp = synthetic.workload_inputs("based_prefill", device=dev)
    y, s, z = la.la_based_prefill(inp["q"], inp["k"], inp["v"])
    torch.cuda.synchronize()
    ref = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")))
    tol = TOL[torch.bfloat16]
    assert rel_err(to_np(y), ref["y"]) < tol
    assert rel_err(to_np(s), ref["s"]) < tol
    assert rel_err(to_np(z), ref["z"]) < tol
    assert la.la_device_status() == la.LA_OK


def test_taylor_output_on_16_byte_boundary():
    """y starting 16 bytes past a 32-byte boundary (rows of 80 bf16): the
    kernel falls back from 32-byte to 16-byte stores; results unchanged."""
    dev = cuda_device()
    inp = synthetic.taylor_inputs(1, 2, 300, dtype=torch.bfloat16, seed=41)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    buf = torch.zeros((1, 2, 300, 80), dtype=torch.bfloat16, device=dev)
    y = buf[..., 8:72]
    _, s, z = la.la_based_prefill(q, k, v, y=y)
    y_ref, s_ref, z_ref = la.la_based_prefill(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref) and torch.equal(s, s_ref) and torch.equal(z, z_ref)
    assert torch.count_nonzero(buf[..., :8]).item() == 0 and torch.count_nonzero(buf[..., 72:]).item() == 0
