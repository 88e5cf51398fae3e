"""The allocation-free gated-delta-rule prefill (la_gdn_prefill_noalloc).

It serves callers that cannot allocate device memory -- a plug-in inside a
framework that owns all device memory, an engine that reserved its budget up
front, a loop that must not pay cudaMalloc's device-wide synchronisation.
Its scratch is a fixed 16 MiB array inside the library, so its results must
match la_gdn_prefill (which takes a caller workspace) on calls that use that
scratch, call after call, while the array keeps the previous call's bytes.

This file is collected last on purpose: it must pass in a fresh process and
after every other test.
"""
import ctypes

import pytest
import torch

import linear_attention_recurrence_chunked_gb300 as la
from tests.helpers import TOL, cuda_device, rel_err, to_np

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "alpha", "beta")


def _inputs(seed, N, dev):
    import synthetic
    x = synthetic.gdn_inputs(1, 2, N, dtype=torch.bfloat16, seed=seed)
    g = torch.Generator().manual_seed(seed)
    # slow decay so the segment maps held in the scratch matter
    x["alpha"] = torch.exp(-(0.001 + 0.001 * torch.rand(x["alpha"].shape, generator=g))).contiguous()
    return {n: x[n].to(dev) for n in NAMES}


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    dev = cuda_device()
    lib = la.load_library()
    tol = TOL[torch.bfloat16]
    for seed, N in ((501, 6144), (502, 7990)):
        x = _inputs(seed, N, dev)
        need_min = la.la_gdn_prefill_workspace_size_min(*(x[n] for n in NAMES))
        assert 0 < need_min <= 16 << 20, "this problem must use segment scratch that fits the fixed array"
        # existing entry point, caller-provided workspace
        o_ref, S_ref = la.la_gdn_prefill(*(x[n] for n in NAMES))
        # new entry point, called straight through the C ABI with caller-owned outputs
        o = torch.empty_like(o_ref)
        S = torch.empty_like(S_ref)
        a = la._gdn_args(x["q"], x["k"], x["v"], o, x["alpha"], x["beta"], None, S, 1.0)
        st = lib.la_gdn_prefill_noalloc(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == la.LA_OK, la.la_status_string(st)
        torch.cuda.synchronize()
        assert rel_err(to_np(o), to_np(o_ref)) < tol
        assert rel_err(to_np(S), to_np(S_ref)) < tol
    assert la.la_device_status() == la.LA_OK


def test_noalloc_refuses_problems_beyond_its_scratch():
    cuda_device()
    lib = la.load_library()
    # 16 heads x 1M tokens needs 25 MiB of segment scratch: refused before any launch
    # (placeholder pointers: nothing is dereferenced when the call is refused)
    B, H, N = 1, 16, 1 << 20
    t = lambda off: la.LATensor(0x100000 + off, H * N * 128, N * 128, 128)
    gt = lambda off: la.LATensor(0x100000 + off, H * N, N, 1)
    a = la.GdnPrefillArgs(B, H, N, 128, 128, la.LA_DTYPE_BF16, la.LA_DTYPE_BF16, t(0), t(1 << 30), t(2 << 30),
                          t(3 << 30), gt(4 << 30), gt(5 << 30), 1.0, None, 0x100000 + (6 << 30))
    assert lib.la_gdn_prefill_workspace_size(ctypes.byref(a)) > 16 << 20
    assert lib.la_gdn_prefill_noalloc(ctypes.byref(a), None) == la.LA_ERR_WORKSPACE
