"""GPU parity of the gated-delta-rule prefill against the fp64 oracle."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "alpha", "beta")


def oracle_ref(inp, S_in=None, q_scale=1.0, t_samples=None):
    return oracle.gdn(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")), inp["alpha"].cpu().numpy(),
                      inp["beta"].cpu().numpy(), S_in=None if S_in is None else S_in.double().cpu().numpy(),
                      q_scale=q_scale, t_samples=t_samples)


def run(inp, dev, **kw):
    o, S = la.la_gdn_prefill(*(inp[n].to(dev) for n in NAMES), **kw)
    torch.cuda.synchronize()
    return to_np(o), to_np(S)


def test_gdn_fp32_small_with_state_in():
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 2, 200, dtype=torch.float32, seed=41)
    S_in = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(4)) * 0.1
    o, S = run(inp, dev, S_in=S_in.to(dev))
    ref = oracle_ref(inp, S_in=S_in)
    assert rel_err(o, ref["o"]) < TOL[torch.float32]
    assert rel_err(S, ref["S"]) < TOL[torch.float32]


@pytest.mark.parametrize("N", [1, 15, 63, 64, 65, 127, 128, 129, 257, 1000])
def test_gdn_bf16_ragged_lengths(N):
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 3, N, dtype=torch.bfloat16, seed=200 + N)
    o, S = run(inp, dev)
    ref = oracle_ref(inp)
    assert rel_err(o, ref["o"]) < TOL[torch.bfloat16]
    assert rel_err(S, ref["S"]) < TOL[torch.bfloat16]


def test_gdn_q_scale_strided_views_fp32_output():
    dev = cuda_device()
    B, H, N = 2, 2, 150
    inp = synthetic.gdn_inputs(B, H, N, dtype=torch.bfloat16, seed=42)
    packed = torch.cat([inp["q"], inp["k"], inp["v"]], dim=-1).permute(0, 2, 1, 3).contiguous().to(dev)
    qv, kv, vv = (packed[..., i * 128:(i + 1) * 128].permute(0, 2, 1, 3) for i in range(3))
    gates = torch.stack([inp["alpha"], inp["beta"]], dim=0).to(dev)  # [2, B, H, N]
    obuf = torch.empty((B, N, H, 128), dtype=torch.float32, device=dev)
    o = obuf.permute(0, 2, 1, 3)
    _, S = la.la_gdn_prefill(qv, kv, vv, gates[0], gates[1], o=o, q_scale=0.5)
    torch.cuda.synchronize()
    ref = oracle_ref(inp, q_scale=0.5)
    assert rel_err(to_np(o), ref["o"]) < TOL[torch.bfloat16]
    assert rel_err(to_np(S), ref["S"]) < TOL[torch.bfloat16]


def test_gdn_split_resume_and_inplace_state():
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 2, 300, dtype=torch.bfloat16, seed=43)
    x = {n: inp[n].to(dev) for n in NAMES}
    o, S = la.la_gdn_prefill(*(x[n] for n in NAMES), out_dtype=torch.float32)
    first = {n: x[n][:, :, :111] for n in NAMES}
    rest = {n: x[n][:, :, 111:] for n in NAMES}
    o1, S1 = la.la_gdn_prefill(*(first[n] for n in NAMES), out_dtype=torch.float32)
    o2, S2 = la.la_gdn_prefill(*(rest[n] for n in NAMES), S_in=S1, S_out=S1, out_dtype=torch.float32)  # in place
    assert S2.data_ptr() == S1.data_ptr()
    # the split moves chunk boundaries, so bf16 operand rounding differs:
    # each run meets the bf16 contract against the oracle, and the two GPU
    # runs agree to well inside it
    ref = oracle_ref(inp)
    o12 = to_np(torch.cat([o1, o2], dim=2))
    assert rel_err(o12, ref["o"]) < TOL[torch.bfloat16] and rel_err(to_np(o), ref["o"]) < TOL[torch.bfloat16]
    assert rel_err(to_np(S2), ref["S"]) < TOL[torch.bfloat16]
    assert rel_err(o12, to_np(o)) < 1e-2
    assert rel_err(to_np(S2), to_np(S)) < 1e-2


def test_gdn_prefill_then_decode_matches_longer_prefill():
    dev = cuda_device()
    inp = synthetic.gdn_inputs(2, 2, 129, dtype=torch.bfloat16, seed=44)
    x = {n: inp[n].to(dev) for n in NAMES}
    _, S = la.la_gdn_prefill(*(x[n][:, :, :128] for n in NAMES))
    o_dec = la.la_decode_step(la.LA_VARIANT_GDN, *(x[n][:, :, 128].contiguous() for n in ("q", "k", "v")), S,
                              alpha=x["alpha"][:, :, 128].contiguous(), beta=x["beta"][:, :, 128].contiguous())
    ref = oracle_ref(inp, t_samples=[128])
    assert rel_err(to_np(o_dec), ref["o"][:, :, 0]) < TOL[torch.bfloat16]
    assert rel_err(to_np(S), ref["S"]) < TOL[torch.bfloat16]


@pytest.mark.parametrize("fn", ["la_gdn_prefill", "la_gated_prefill"])
def test_records_formed_beside_the_scan_match_the_inversion_kernel(fn):
    """With few enough (b,h) pairs (unsegmented sequences), the chunk records
    are formed in the scan's own launch, on the SMs its scan CTAs leave free,
    and handed over through per-record flags; with more pairs a separate
    inversion kernel forms them first.  Both use the same arithmetic, so the
    first 64 pairs of a 144-pair call give exactly the bits of a 64-pair call
    on the same inputs; two heads of the large call are checked against the
    oracle."""
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 144, 700, dtype=torch.bfloat16, seed=47)
    f = getattr(la, fn)
    x = {n: inp[n].to(dev) for n in NAMES}
    o_all, S_all = f(*(x[n] for n in NAMES))
    o_64, S_64 = f(*(x[n][:, :64].contiguous() for n in NAMES))
    torch.cuda.synchronize()
    assert la.la_device_status() == la.LA_OK
    assert torch.equal(o_all[:, :64], o_64) and torch.equal(S_all[:, :64], S_64)
    heads = [5, 130]
    sub = {n: inp[n][:, heads] for n in NAMES}
    ref = (oracle.gdn if fn == "la_gdn_prefill" else oracle.gated)(
        *(synthetic.to_oracle(sub[n]) for n in ("q", "k", "v")), sub["alpha"].numpy(), sub["beta"].numpy())
    assert rel_err(to_np(o_all[:, heads]), ref["o"]) < TOL[torch.bfloat16]
    assert rel_err(to_np(S_all[:, heads]), ref["S"]) < TOL[torch.bfloat16]


def test_one_launch_at_its_largest_pair_count():
    """The one-launch schedule runs while the (b,h) pairs leave at least 16 of the
    GPU's SMs for forming the records: at that limit only 16 record-forming CTAs
    serve every pair, and their pacing lead (three times their record spacing)
    is a single chunk.  Its results are the bits of the same pairs run with the
    records from the chunk-parallel kernel (one more pair than the limit), and two
    heads meet the oracle."""
    dev = cuda_device()
    limit = torch.cuda.get_device_properties(dev).multi_processor_count - 16
    inp = synthetic.gdn_inputs(1, limit + 1, 1000, dtype=torch.bfloat16, seed=53)
    x = {n: inp[n].to(dev) for n in NAMES}
    o_two, S_two = la.la_gdn_prefill(*(x[n] for n in NAMES))          # limit + 1 pairs: two kernels
    o_one, S_one = la.la_gdn_prefill(*(x[n][:, :limit].contiguous() for n in NAMES))  # one launch
    torch.cuda.synchronize()
    assert la.la_device_status() == la.LA_OK
    assert torch.equal(o_two[:, :limit], o_one) and torch.equal(S_two[:, :limit], S_one)
    heads = [0, limit - 1]
    sub = {n: inp[n][:, heads] for n in NAMES}
    ref = oracle.gdn(*(synthetic.to_oracle(sub[n]) for n in ("q", "k", "v")), sub["alpha"].numpy(),
                     sub["beta"].numpy())
    assert rel_err(to_np(o_one[:, heads]), ref["o"]) < TOL[torch.bfloat16]
    assert rel_err(to_np(S_one[:, heads]), ref["S"]) < TOL[torch.bfloat16]


def test_gdn_empty_sequence_passes_state():
    dev = cuda_device()
    z = torch.zeros((1, 2, 0, 128), dtype=torch.bfloat16, device=dev)
    g = torch.zeros((1, 2, 0), dtype=torch.float32, device=dev)
    S_in = torch.randn((1, 2, 128, 128), device=dev)
    _, S = la.la_gdn_prefill(z, z, z, g, g, S_in=S_in)
    assert torch.equal(S, S_in)


def test_gdn_prefill_full_size():
    """Gated DeltaNet prefill bf16/fp32-state: B=4, H=16, N=16384, the launch
    the benchmark times; every head checked against the oracle on every token
    and every state entry (max-normalised and floored elementwise errors)."""
    dev = cuda_device()
    w = synthetic.WORKLOADS["gdn_prefill"]
    inp = synthetic.workload_inputs("gdn_prefill", device=dev)
    o, S = la.la_gdn_prefill(*(inp[n] for n in NAMES))
    torch.cuda.synchronize()
    tol = TOL[torch.bfloat16]
    assert la.la_device_status() == la.LA_OK
    for b in range(w.B):  # one batch row (16 heads) of oracle work at a time
        sub = {n: inp[n][b:b + 1].cpu() for n in NAMES}
        ref = oracle_ref(sub)
        assert rel_err(to_np(o[b:b + 1]), ref["o"]) < tol, b
        assert rel_err(to_np(S[b:b + 1]), ref["S"]) < tol, b


def test_gdn_prefill_long_context_full_size():
    """Long-context Gated DeltaNet prefill: B=1, H=16, N=1,048,576.  The whole
    launch runs on the GPU; two heads are recomputed by the oracle over all
    1M tokens and compared on 64 sampled output positions and the final state."""
    dev = cuda_device()
    w = synthetic.WORKLOADS["gdn_prefill_long"]
    inp = synthetic.workload_inputs("gdn_prefill_long", device=dev)
    o, S = la.la_gdn_prefill(*(inp[n] for n in NAMES))
    torch.cuda.synchronize()
    heads = [3, 12]
    rng = np.random.default_rng(8)
    t_samples = np.unique(np.concatenate([rng.choice(w.N, 60, replace=False), [0, 1, w.N - 2, w.N - 1]]))
    sub = {n: inp[n][:, heads].cpu() for n in NAMES}
    ref = oracle_ref(sub, t_samples=t_samples)
    tol = TOL[torch.bfloat16]
    ts = torch.tensor(t_samples, device=dev)
    assert rel_err(to_np(o[:, heads][:, :, ts]), ref["o"]) < tol
    assert rel_err(to_np(S[:, heads]), ref["S"]) < tol
    del inp, o
    assert la.la_device_status() == la.LA_OK


def _slow_decay(inp, seed):
    """alpha close to 1 (exp(-U(0.001, 0.002))): a 2048-token segment keeps a
    sizeable part of its entry state, so the segment maps are far from zero."""
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(inp["alpha"].shape, generator=g)
    inp = dict(inp)
    inp["alpha"] = torch.exp(-(0.001 + 0.001 * u)).contiguous()
    return inp


@pytest.mark.parametrize("N,inplace", [(6144, False), (7990, True)])
def test_gdn_sequence_segments_match_oracle(N, inplace):
    """Few heads and a long sequence take the segment path (maps per segment,
    a combine, then all segments in parallel); results must match the oracle."""
    dev = cuda_device()
    inp = _slow_decay(synthetic.gdn_inputs(1, 2, N, dtype=torch.bfloat16, seed=300 + N), seed=N)
    x = {n: inp[n].to(dev) for n in NAMES}
    assert la.la_gdn_prefill_workspace_size_min(*(x[n] for n in NAMES)) > 0, "expected the segment path"
    S_in = (torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(9)) * 0.1)
    S_dev = S_in.to(dev).contiguous()
    o, S = la.la_gdn_prefill(*(x[n] for n in NAMES), S_in=S_dev, S_out=S_dev if inplace else None)
    torch.cuda.synchronize()
    ref = oracle_ref(inp, S_in=S_in)
    tol = TOL[torch.bfloat16]
    assert rel_err(to_np(o), ref["o"]) < tol
    assert rel_err(to_np(S), ref["S"]) < tol
    assert la.la_device_status() == la.LA_OK


@pytest.mark.parametrize("B,H,N,seg", [(1, 3, 1000, False), (2, 2, 257, False), (1, 2, 6144, True)])
def test_gdn_two_schedules_agree(B, H, N, seg):
    """The records schedule (chunk records, then the state chain) and
    the one-kernel scan compute the same chunk form; they differ only in
    where roundings fall (the chain keeps S / sigma with a running decay
    sigma, and rounds q_scale diag(gamma) Q to bf16), so they must agree far
    inside the bf16 tolerance -- with an incoming state, fp32 outputs, and on
    the segment path too.  Both are also checked against the oracle."""
    dev = cuda_device()
    inp = synthetic.gdn_inputs(B, H, N, dtype=torch.bfloat16, seed=600 + N)
    if seg:
        inp = _slow_decay(inp, seed=N)
    x = {n: inp[n].to(dev) for n in NAMES}
    need = la.la_gdn_prefill_workspace_size(*(x[n] for n in NAMES))
    need_min = la.la_gdn_prefill_workspace_size_min(*(x[n] for n in NAMES))
    assert need > need_min and (need_min > 0) == seg
    S_in = torch.randn((B, H, 128, 128), generator=torch.Generator().manual_seed(N)) * 0.1
    outs = []
    for ws_bytes in (need, need_min):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        o, S = la.la_gdn_prefill(*(x[n] for n in NAMES), S_in=S_in.to(dev), out_dtype=torch.float32, workspace=ws)
        torch.cuda.synchronize()
        outs.append((o.cpu(), S.cpu()))
    ref = oracle_ref(inp, S_in=S_in)
    tol = TOL[torch.bfloat16]
    for o, S in outs:
        assert rel_err(o.numpy(), ref["o"]) < tol
        assert rel_err(S.numpy(), ref["S"]) < tol
    assert rel_err(outs[0][0].numpy(), outs[1][0].numpy().astype(np.float64)) < 5e-3
    assert rel_err(outs[0][1].numpy(), outs[1][1].numpy().astype(np.float64)) < 5e-3
    assert la.la_device_status() == la.LA_OK


def test_gdn_workspace_between_min_and_full_runs_one_kernel_schedule():
    """A workspace one byte short of the records schedule's need still runs (one-kernel
    schedule); a misaligned one is refused without a launch."""
    dev = cuda_device()
    inp = synthetic.gdn_inputs(1, 2, 300, dtype=torch.bfloat16, seed=71)
    x = {n: inp[n].to(dev) for n in NAMES}
    need = la.la_gdn_prefill_workspace_size(*(x[n] for n in NAMES))
    ws = torch.empty(need + 16, dtype=torch.uint8, device=dev)
    o1, S1 = la.la_gdn_prefill(*(x[n] for n in NAMES), workspace=ws[: need - 1])
    o2, S2 = la.la_gdn_prefill(*(x[n] for n in NAMES), workspace=ws[:need])
    torch.cuda.synchronize()
    assert rel_err(to_np(o1), to_np(o2)) < 5e-3 and rel_err(to_np(S1), to_np(S2)) < 5e-3
    with pytest.raises(la.LAError):
        la.la_gdn_prefill(*(x[n] for n in NAMES), workspace=ws[1:need + 1])
    assert la.la_device_status() == la.LA_OK
