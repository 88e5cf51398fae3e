"""GPU parity of the state operations between calls (NoteBank App. D.1
readout-boundary rescale/reset; App. B Alg. 1 state copy) against their
plain definitions: one fp32 multiplication or a copy per element, so the
comparison is bit-exact."""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,state_dims", [((3, 4, 128, 128), 2), ((2, 5, 273, 64), 2), ((2, 5, 273), 1),
                                              ((7, 3, 5), 1)])
def test_rescale_bit_exact_scalar_and_per_state(shape, state_dims):
    dev = cuda_device()
    g = torch.Generator().manual_seed(sum(shape))
    S = torch.randn(shape, generator=g)
    lead = shape[: len(shape) - state_dims]
    lam = torch.rand(lead, generator=g)
    lam.view(-1)[0] = 0.0  # one reset among them
    x = S.to(dev)
    la.la_state_rescale(x, lam.to(dev).contiguous(), state_dims=state_dims)
    assert np.array_equal(to_np(x), oracle.state_rescale(S.numpy(), lam.numpy(), state_dims))
    y = S.to(dev)
    la.la_state_rescale(y, 0.3, state_dims=state_dims)
    assert np.array_equal(to_np(y), oracle.state_rescale(S.numpy(), np.float32(0.3), state_dims))


def test_reset_clears_non_finite_state_and_scalar_path_on_4_byte_alignment():
    dev = cuda_device()
    buf = torch.randn(4 * 1000 + 1, device=dev)
    buf[5] = float("nan")
    buf[17] = float("inf")
    view = buf[1:].view(4, 1000)  # 4-byte aligned only: the scalar path
    la.la_state_rescale(view, 0.0, state_dims=1)
    torch.cuda.synchronize()
    assert torch.count_nonzero(view).item() == 0
    assert torch.isfinite(buf[0]).item()  # the element before the view is untouched


def test_gather_copies_branches_and_skips_bad_indices():
    dev = cuda_device()
    g = torch.Generator().manual_seed(4)
    src = torch.randn((6, 128, 128), generator=g)
    idx = torch.tensor([5, 0, 5, 5, 2], dtype=torch.int64)
    out = la.la_state_gather(src.to(dev), idx.to(dev))
    assert np.array_equal(to_np(out), oracle.state_gather(src.numpy(), idx.tolist()))
    assert la.la_device_status() == la.LA_OK
    # Taylor z rows (273 floats: the scalar path)
    z = torch.rand((4, 273), generator=g)
    zo = la.la_state_gather(z.to(dev), torch.tensor([3, 1], dtype=torch.int64, device=dev), state_dims=1)
    assert np.array_equal(to_np(zo), oracle.state_gather(z.numpy(), [3, 1], state_dims=1))
    # an out-of-range index leaves its destination untouched and is reported
    dst = torch.full((3, 128, 128), 7.0, device=dev)
    la.la_state_gather(src.to(dev), torch.tensor([1, 6, -1], dtype=torch.int64, device=dev), dst=dst)
    assert la.la_device_status() == la.LA_ERR_INVALID_ARGUMENT
    assert np.array_equal(to_np(dst[0]), src[1].numpy())
    assert torch.all(dst[1:] == 7.0).item()
    assert la.la_device_status() == la.LA_OK  # cleared by the previous read
    # overlapping source and destination are refused before any launch
    with pytest.raises(la.LAError):
        la.la_state_gather(dst, torch.tensor([0], dtype=torch.int64, device=dev), dst=dst[1:2])


def test_branch_rescale_and_replay_against_oracle():
    """The NoteBank sequence on one GDN head: prefill the context, copy the
    state to a branch, reset the branch (lambda = 0) and rescale the original
    (lambda = 0.5), then continue both with the same replay tokens; each
    branch must match the oracle run from the same entry state."""
    dev = cuda_device()
    ctx = synthetic.gdn_inputs(1, 2, 500, dtype=torch.bfloat16, seed=91)
    rep = synthetic.gdn_inputs(1, 2, 130, dtype=torch.bfloat16, seed=92)
    names = ("q", "k", "v", "alpha", "beta")
    _, S = la.la_gdn_prefill(*(ctx[n].to(dev) for n in names))
    branch = la.la_state_gather(S.view(2, 128, 128), torch.tensor([0, 1], dtype=torch.int64, device=dev)).view(1, 2, 128, 128)
    la.la_state_rescale(branch, 0.0)
    la.la_state_rescale(S, 0.5)
    S_host = to_np(S)
    tol = TOL[torch.bfloat16]
    for entry, entry_host in ((branch, np.zeros_like(S_host)), (S, S_host)):
        o, S_end = la.la_gdn_prefill(*(rep[n].to(dev) for n in names), S_in=entry)
        ref = oracle.gdn(*(synthetic.to_oracle(rep[n]) for n in ("q", "k", "v")), rep["alpha"].numpy(),
                         rep["beta"].numpy(), S_in=entry_host)
        assert rel_err(to_np(o), ref["o"]) < tol
        assert rel_err(to_np(S_end), ref["S"]) < tol
    assert la.la_device_status() == la.LA_OK
