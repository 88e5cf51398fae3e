"""The allocation-free gated-delta-rule prefill (la_gdn_prefill_noalloc).

It serves callers that cannot allocate device memory -- a plug-in inside a
framework that owns all device memory, an engine that reserved its budget up
front, a loop that must not pay cudaMalloc's device-wide synchronisation.
Its scratch is a fixed 16 MiB array inside the library, shared by every call
and keeping the previous call's bytes.  So its results must equal, bit for
bit, those of la_gdn_prefill (which takes a caller workspace and runs the same
schedule on these problems) on two different problems in a row, and meet the
fp64 oracle; and the calls must not change the device's free memory.

This file is collected last on purpose: it must pass in a fresh process and
after every other test.
"""
import ctypes

import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
import oracle
import synthetic
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "alpha", "beta")


def _inputs(seed, N):
    x = synthetic.gdn_inputs(1, 2, N, dtype=torch.bfloat16, seed=seed)
    g = torch.Generator().manual_seed(seed)
    # slow decay so the segment maps held in the scratch matter
    x["alpha"] = torch.exp(-(0.001 + 0.001 * torch.rand(x["alpha"].shape, generator=g))).contiguous()
    return x


def _oracle(x, S_in=None):
    return oracle.gdn(*(synthetic.to_oracle(x[n]) for n in ("q", "k", "v")), x["alpha"].numpy(), x["beta"].numpy(),
                      S_in=None if S_in is None else S_in.double().cpu().numpy())


def _call_c_abi(lib, xd, o, S, S_in=None):
    a = la._gdn_args(xd["q"], xd["k"], xd["v"], o, xd["alpha"], xd["beta"], S_in, S, 1.0)
    return lib.la_gdn_prefill_noalloc(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    dev = cuda_device()
    lib = la.load_library()
    tol = TOL[torch.bfloat16]
    problems = [(501, 6144), (502, 7990)]  # different sizes and data: stale scratch would show
    xs = [_inputs(seed, N) for seed, N in problems]
    xds = [{n: x[n].to(dev) for n in NAMES} for x in xs]
    refs = []
    for xd in xds:
        args = [xd[n] for n in NAMES]
        need_min = la.la_gdn_prefill_workspace_size_min(*args)
        need = la.la_gdn_prefill_workspace_size(*args)
        # segment scratch and per-chunk records both fit the fixed array, so both entry
        # points run the same records schedule with segments
        assert 0 < need_min <= need <= 16 << 20
        refs.append(la.la_gdn_prefill(*args))  # existing entry point, caller workspace
    outs = [(torch.empty_like(o), torch.empty_like(S)) for o, S in refs]
    # warm-up call: kernels loaded, the array's address looked up
    assert _call_c_abi(lib, xds[0], *outs[0]) == la.LA_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(dev)[0]
    for xd, (o, S) in zip(xds, outs):
        st = _call_c_abi(lib, xd, o, S)
        assert st == la.LA_OK, la.la_status_string(st)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free_before, "the no-alloc calls changed the device's free memory"
    for x, (o_ref, S_ref), (o, S) in zip(xs, refs, outs):
        assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
        assert rel_err(to_np(o), to_np(o_ref)) < tol and rel_err(to_np(S), to_np(S_ref)) < tol
        ref = _oracle(x)
        assert rel_err(to_np(o), ref["o"]) < tol
        assert rel_err(to_np(S), ref["S"]) < tol
    assert la.la_device_status() == la.LA_OK


def test_noalloc_python_wrapper_with_incoming_state():
    dev = cuda_device()
    tol = TOL[torch.bfloat16]
    x = _inputs(503, 3000)
    xd = {n: x[n].to(dev) for n in NAMES}
    S_in = torch.randn((1, 2, 128, 128), generator=torch.Generator().manual_seed(7)) * 0.1
    o_ref, S_ref = la.la_gdn_prefill(*(xd[n] for n in NAMES), S_in=S_in.to(dev))
    o = torch.empty_like(o_ref)
    S = torch.empty_like(S_ref)
    la.la_gdn_prefill_noalloc(*(xd[n] for n in NAMES), o, S, S_in=S_in.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
    ref = _oracle(x, S_in=S_in)
    assert rel_err(to_np(o), ref["o"]) < tol
    assert rel_err(to_np(S), ref["S"]) < tol


def test_noalloc_refuses_problems_beyond_its_scratch():
    cuda_device()
    lib = la.load_library()
    # placeholder pointers: nothing is dereferenced when a call is refused
    def args(H, N):
        t = lambda off: la.LATensor(0x100000 + off, H * N * 128, N * 128, 128)
        gt = lambda off: la.LATensor(0x100000 + off, H * N, N, 1)
        return la.GdnPrefillArgs(1, H, N, 128, 128, la.LA_DTYPE_BF16, la.LA_DTYPE_BF16, t(0), t(1 << 30),
                                 t(2 << 30), t(3 << 30), gt(4 << 30), gt(5 << 30), 1.0, None, 0x100000 + (6 << 30))
    # 16 heads x 1M tokens: 9 segments per head, 16 x (2 x 8 + 9) fp32 128x128 blocks = 25 MiB of
    # segment scratch, beyond the 16 MiB array: refused before any launch
    a = args(16, 1 << 20)
    assert lib.la_gdn_prefill_workspace_size_min(ctypes.byref(a)) == 16 * (2 * 8 + 9) * 128 * 128 * 4 == 26214400
    assert lib.la_gdn_prefill_noalloc(ctypes.byref(a), None) == la.LA_ERR_WORKSPACE
