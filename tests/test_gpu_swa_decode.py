"""GPU parity of the sliding-window softmax-attention decode step (the window
layers of BASED, BASED notes Sec. 2.4-2.5) against the fp64 oracle.

Sequences start at different positions: their ring buffers are filled by the
test with the tokens before the first step (token p in slot p % window), so
every step mixes full and still-filling windows and wraps around the ring."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu


def _draw(S, H, N, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((S, H, N, d), generator=g) / d ** 0.25).to(dtype)
    k = (torch.randn((S, H, N, d), generator=g) / d ** 0.25).to(dtype)
    v = torch.randn((S, H, N, d), generator=g).to(dtype)
    return q, k, v


@pytest.mark.parametrize("window,d,dtype", [(64, 64, torch.bfloat16), (16, 64, torch.bfloat16),
                                            (128, 128, torch.bfloat16), (1, 64, torch.float32),
                                            (64, 64, torch.float32), (256, 32, torch.bfloat16),
                                            (256, 128, torch.bfloat16), (256, 128, torch.float32)])
def test_swa_decode_matches_oracle(window, d, dtype):
    """d of 64 or 128 stages each window in shared memory (four warps per CTA, or fewer for large
    windows: one for 256 x 128 bf16); d = 32 and 256 x 128 fp32 (too large) take the direct kernel."""
    dev = cuda_device()
    S, H, steps = 5, 3, 40
    offsets = [0, 3, window - 1, window + 5, 3 * window + 2]
    N = steps + max(offsets)
    q, k, v = _draw(S, H, N, d, dtype, seed=window * 7 + d)
    kc = torch.zeros((S, H, window, d), dtype=dtype)
    vc = torch.zeros((S, H, window, d), dtype=dtype)
    for s, off in enumerate(offsets):  # tokens before the first step, in their ring slots
        for p in range(max(0, off - window), off):
            kc[s, :, p % window] = k[s, :, p]
            vc[s, :, p % window] = v[s, :, p]
    kc, vc = kc.to(dev), vc.to(dev)
    scale = d ** -0.5
    ref = [oracle.swa(synthetic.to_oracle(q[s:s + 1]), synthetic.to_oracle(k[s:s + 1]),
                      synthetic.to_oracle(v[s:s + 1]), window, scale,
                      t_samples=list(range(offsets[s], offsets[s] + steps)))[0] for s in range(S)]
    ref = np.stack(ref)  # [S, H, steps, d]
    outs = []
    for t in range(steps):
        pos = torch.tensor([off + t for off in offsets], dtype=torch.int64, device=dev)
        idx = pos.cpu()
        qt = torch.stack([q[s, :, idx[s]] for s in range(S)]).to(dev).contiguous()
        kt = torch.stack([k[s, :, idx[s]] for s in range(S)]).to(dev).contiguous()
        vt = torch.stack([v[s, :, idx[s]] for s in range(S)]).to(dev).contiguous()
        outs.append(to_np(la.la_swa_decode_step(qt, kt, vt, kc, vc, pos)))
    got = np.stack(outs, axis=2)
    assert rel_err(got, ref) < TOL[dtype]
    assert la.la_device_status() == la.LA_OK


def test_swa_decode_negative_position_is_reported_and_skipped():
    dev = cuda_device()
    S, H, d, window = 2, 2, 64, 16
    q, k, v = (torch.randn((S, H, d), device=dev) for _ in range(3))
    kc = torch.full((S, H, window, d), 3.0, device=dev)
    vc = torch.full((S, H, window, d), 3.0, device=dev)
    out = torch.full((S, H, d), -1.0, device=dev)
    pos = torch.tensor([-4, 0], dtype=torch.int64, device=dev)
    la.la_swa_decode_step(q, k, v, kc, vc, pos, out=out)
    assert la.la_device_status() == la.LA_ERR_INVALID_ARGUMENT
    assert torch.all(out[0] == -1.0).item() and torch.all(kc[0] == 3.0).item()  # untouched
    assert torch.allclose(out[1], v[1], atol=1e-6)  # pos 0: the window holds only the new token
    assert torch.equal(kc[1, :, 0], k[1])


def test_swa_decode_full_size_sampled():
    """The benchmark's launch: 256 sequences x 16 heads, window 64, d 64, bf16, every ring full at the
    first step; 8 steps, 16 sampled (sequence, head) pairs against the oracle at every step."""
    dev = cuda_device()
    S, H, window, d, steps = 256, 16, 64, 64, 8
    # tokens 0..63 are already in the rings (token p in slot p); tokens 64..71 arrive one per step
    q_all, k_all, v_all = _draw(S, H, window + steps, d, torch.bfloat16, seed=21)
    kc = k_all[:, :, :window].contiguous().to(dev)
    vc = v_all[:, :, :window].contiguous().to(dev)
    scale = d ** -0.5
    outs = []
    for t in range(steps):
        p = window + t
        pos = torch.full((S,), p, dtype=torch.int64, device=dev)
        outs.append(la.la_swa_decode_step(*(x[:, :, p].contiguous().to(dev) for x in (q_all, k_all, v_all)),
                                          kc, vc, pos, scale=scale))
    got = torch.stack(outs, dim=2)  # [S, H, steps, d]
    rng = np.random.default_rng(5)
    pairs = sorted(rng.choice(S * H, 16, replace=False).tolist())
    si, hi = [p // H for p in pairs], [p % H for p in pairs]

    def sub(x):  # [1, pairs, tokens, d]
        return torch.stack([x[s, h] for s, h in zip(si, hi)]).unsqueeze(0)

    ref = oracle.swa(*(synthetic.to_oracle(sub(x)) for x in (q_all, k_all, v_all)), window, scale,
                     t_samples=list(range(window, window + steps)))
    assert rel_err(to_np(sub(got.cpu())), ref) < TOL[torch.bfloat16]
    assert la.la_device_status() == la.LA_OK
