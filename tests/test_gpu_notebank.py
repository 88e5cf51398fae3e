"""GPU parity of NoteBank's write side and routing (NoteBank Sec. 2 Eqs. (3)-(5),
App. B Eqs. (8)-(9)) against the oracle.

Scores are compared within fp32 rounding.  Where floating point decides an
integer (an argmax), both sides decide in the kernel's precision: the
address oracle is fed the kernel's own fp32 scores, so t* and the gathered
bf16 addresses must match exactly; for routing the kernel's winners must be
valid (a maximum of the oracle's fp32 cosines up to rounding), and the votes
and the retrieved notes must follow exactly from those winners."""
import json
import os

import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import cuda_device, to_np

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def keys(L, H, N, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((L, H, N, d), generator=g).to(dtype)


@pytest.mark.parametrize("L,H,N,d,chunk,dtype", [(3, 4, 1100, 128, 512, torch.bfloat16),
                                                  (2, 2, 700, 256, 256, torch.bfloat16),
                                                  (1, 3, 333, 32, 100, torch.float32),
                                                  (2, 1, 47, 64, 512, torch.bfloat16),
                                                  (1, 2, 1500, 256, 1024, torch.float32),
                                                  (1, 1, 3, 32, 512, torch.bfloat16)])
def test_scores_match_oracle(L, H, N, d, chunk, dtype):
    """Most shapes keep a chunk's keys in the shared memory of a 4-CTA cluster; fp32
    keys of width 256 in chunks of 1024 do not fit and take two passes over global
    memory; 3 tokens leave three of the cluster's CTAs without rows."""
    dev = cuda_device()
    k = keys(L, H, N, d, dtype, seed=N + d)
    zero = min(5, N - 1)
    k[0, 0, zero] = 0  # a zero key scores 1
    d_ch, d_mean, w = la.la_notebank_scores(k.to(dev), chunk=chunk, window=48)
    ref = oracle.notebank_scores(synthetic.to_oracle(k), chunk=chunk, window=48)
    torch.cuda.synchronize()
    assert np.max(np.abs(to_np(d_ch) - ref["d_ch"])) < 2e-5
    assert np.max(np.abs(to_np(d_mean) - ref["d"])) < 2e-5
    assert w.numel() == ref["w"].size
    if w.numel():
        assert np.max(np.abs(to_np(w) - ref["w"])) < 1e-3
    assert abs(float(d_ch[0, 0, zero]) - 1.0) < 1e-6


def test_scores_strided_channels():
    """k carved out of a [N, L, H, d + 32] buffer (token-major, padded rows)."""
    dev = cuda_device()
    L, H, N, d = 2, 3, 600, 128
    g = torch.Generator().manual_seed(5)
    buf = torch.randn((N, L, H, d + 32), generator=g).to(torch.bfloat16).to(dev)
    k = buf[..., :d].permute(1, 2, 0, 3)
    d_ch, d_mean, w = la.la_notebank_scores(k, chunk=512, window=48)
    ref = oracle.notebank_scores(synthetic.to_oracle(k.contiguous().cpu()), chunk=512, window=48)
    torch.cuda.synchronize()
    assert np.max(np.abs(to_np(d_ch) - ref["d_ch"])) < 2e-5


def test_address_matches_oracle_exactly():
    dev = cuda_device()
    L, H, N, d, n = 2, 3, 900, 128, 11
    k = keys(L, H, N, d, torch.bfloat16, seed=1)
    q = keys(L, H, N, d, torch.bfloat16, seed=2)
    d_ch, _, _ = la.la_notebank_scores(k.to(dev), chunk=512)
    g = torch.Generator().manual_seed(3)
    coords = torch.stack([torch.randperm(d, generator=g)[:16] for _ in range(L * H)]).view(L, H, 16).to(torch.int32)
    starts = torch.randint(0, N - 64, (n,), generator=g)
    lens = torch.randint(1, 65, (n,), generator=g)
    spans = torch.stack([starts, lens], dim=1).to(torch.int64)
    spans[0] = torch.tensor([N - 1, 1])          # the last token alone
    t_star, rho = la.la_notebank_address(d_ch, q.to(dev), coords.to(dev), spans.to(dev))
    torch.cuda.synchronize()
    ref_t, ref_rho = oracle.notebank_address(to_np(d_ch), synthetic.to_oracle(q), coords.numpy(), spans.numpy())
    assert np.array_equal(np.array(t_star.tolist()), ref_t)
    assert np.array_equal(rho.float().cpu().numpy(), ref_rho)
    assert la.la_device_status() == la.LA_OK


def test_address_reports_bad_spans_and_coordinates():
    dev = cuda_device()
    L, H, N, d = 1, 2, 100, 64
    q = keys(L, H, N, d, torch.bfloat16, seed=4).to(dev)
    d_ch = torch.rand((L, H, N), device=dev)
    coords = torch.arange(16, dtype=torch.int32, device=dev).repeat(L, H, 1).contiguous()
    coords[0, 1, 3] = 64  # outside [0, d): channel (0,1) of every note is rejected
    spans = torch.tensor([[10, 5], [98, 5], [-1, 3], [20, 0]], dtype=torch.int64, device=dev)
    t_star, rho = la.la_notebank_address(d_ch, q, coords, spans)
    assert la.la_device_status() == la.LA_ERR_INVALID_ARGUMENT
    ts = np.array(t_star.tolist())
    assert ts[0, 0, 0] == 10 + int(torch.argmax(d_ch[0, 0, 10:15]))
    assert np.all(ts[1:, 0, 0] == -1) and np.all(ts[:, 0, 1] == -1)
    assert torch.count_nonzero(rho[1:]).item() == 0 and torch.count_nonzero(rho[:, 0, 1]).item() == 0
    assert la.la_device_status() == la.LA_OK


def check_route(rho, u, R, positions=None):
    dev = cuda_device()
    top, winner, votes, s = la.la_notebank_route(rho.to(dev), u.to(dev), R,
                                                 positions=None if positions is None else positions.to(dev),
                                                 want_scores=True)
    torch.cuda.synchronize()
    ref = oracle.notebank_route(rho.float().numpy(), u.float().numpy(), R,
                                positions=None if positions is None else positions.numpy())
    assert np.max(np.abs(to_np(s) - ref["s"])) < 1e-5
    w = np.array(winner.tolist(), dtype=np.int64)
    for j, wj in enumerate(w):  # a valid maximum of the oracle's cosines
        assert ref["s"][wj, j] >= ref["s"][:, j].max() - 1e-5
    n = rho.shape[0]
    assert np.array_equal(np.array(votes.tolist()), np.bincount(w, minlength=n))
    # the retrieved notes follow exactly from the kernel's votes
    v = np.bincount(w, minlength=n)
    order = sorted((i for i in range(n) if v[i] >= 1), key=lambda i: (-v[i], i))[:R]
    pos = np.arange(n) if positions is None else positions.numpy()
    want = sorted(order, key=lambda i: (pos[i], i)) + [-1] * (R - len(order))
    assert top.tolist() == want
    return w, ref


def test_route_random_notes():
    g = torch.Generator().manual_seed(8)
    n, J, nq, R = 300, 48, 20, 4
    rho = torch.randn((n, J, 16), generator=g).to(torch.bfloat16)
    u = torch.randn((J, nq, 16), generator=g).to(torch.bfloat16)
    positions = torch.randperm(n, generator=g).to(torch.int64) * 64
    w, ref = check_route(rho, u, R, positions)
    assert np.mean(w == ref["winner"]) > 0.95  # exact agreement except at fp32 near-ties


def test_route_worked_example_and_no_notes():
    g = json.load(open(os.path.join(GOLDEN, "notebank_vote_example.json")))
    names = g["notes"]
    J = len(g["channel_winners"])
    rho = torch.zeros((len(names), J, 16))
    for j, win in enumerate(g["channel_winners"]):
        for i, nm in enumerate(names):
            rho[i, j, j if nm == win else j + 1] = 1.0
    u = torch.zeros((J, 1, 16))
    for j in range(J):
        u[j, 0, j] = 1.0
    dev = cuda_device()
    top, winner, votes, _ = la.la_notebank_route(rho.to(torch.bfloat16).to(dev), u.to(torch.bfloat16).to(dev), g["R"],
                                                 positions=torch.tensor([500, 100], dtype=torch.int64, device=dev))
    assert [names[i] for i in winner.tolist()] == g["channel_winners"]
    assert {names[i]: v for i, v in enumerate(votes.tolist())} == g["votes"]
    assert [names[i] for i in top.tolist()] == ["B", "A"]  # text order, not vote order
    empty = torch.zeros((0, J, 16), dtype=torch.bfloat16, device=dev)
    top, winner, _, _ = la.la_notebank_route(empty, u.to(torch.bfloat16).to(dev), 2)
    assert top.tolist() == [-1, -1] and winner.tolist() == [-1] * J


def test_route_pages_scale_sampled():
    """The pages' scale: 4092 notes, 192 channels, a 64-token question."""
    g = torch.Generator().manual_seed(9)
    n, J, nq = 4092, 192, 64
    rho = torch.randn((n, J, 16), generator=g).to(torch.bfloat16)
    u = torch.randn((J, nq, 16), generator=g).to(torch.bfloat16)
    check_route(rho, u, 2)


def test_scores_full_size():
    """The benchmark's launch: 192 channels (24 layers x 8 heads), 16384 tokens, d_k 256, chunks of 512;
    every channel's scores, the channel mean and the window sums against the oracle (run one layer of
    8 channels at a time; the mean over all channels is the mean of the 24 layers' means)."""
    dev = cuda_device()
    L, H, N, d = 24, 8, 16384, 256
    gen = torch.Generator(device=dev).manual_seed(13)
    k = torch.randn((L, H, N, d), generator=gen, device=dev).to(torch.bfloat16)
    d_ch, d_mean, w = la.la_notebank_scores(k, chunk=512, window=48)
    torch.cuda.synchronize()
    assert la.la_device_status() == la.LA_OK
    d_ch_np = to_np(d_ch)
    layer_means = []
    for l in range(L):
        ref = oracle.notebank_scores(synthetic.to_oracle(k[l:l + 1].cpu()), chunk=512, window=48)
        assert np.max(np.abs(d_ch_np[l:l + 1] - ref["d_ch"])) < 2e-5, l
        layer_means.append(ref["d"])
    d_ref = np.mean(layer_means, axis=0)
    assert np.max(np.abs(to_np(d_mean).astype(np.float64) - d_ref)) < 1e-5
    c = np.concatenate([[0.0], np.cumsum(d_ref)])
    w_ref = c[48:] - c[:-48]
    assert w.numel() == w_ref.size and np.max(np.abs(to_np(w).astype(np.float64) - w_ref)) < 1e-3
