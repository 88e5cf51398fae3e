"""Host-side checks of the C ABI: the library loads without a GPU, exports
every entry point include/la.h declares, and rejects malformed arguments with
status codes before any CUDA call (only argument validation runs here)."""
import ctypes
import os
import re
import subprocess

import pytest

import linear_attention_recurrence_chunked_gb300 as la
from linear_attention_recurrence_chunked_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return la.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(la_[a-z0-9_]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"la_based_prefill", "la_gdn_prefill", "la_decode_step"} <= names
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (la_[a-z0-9_]+)\b", out))
    assert names <= exported, f"missing exports: {names - exported}"
    for n in names:
        assert hasattr(lib, n)
    assert set(la.EXPORTED) <= names


def test_abi_version_and_status_strings(lib):
    assert la.la_abi_version() == 2
    for code in range(6):
        assert la.la_status_string(code)
    assert la.la_status_string(99) == "unknown status"


def _tensor(ptr, sb=0, sh=0, st=0):
    return la.LATensor(ptr, sb, sh, st)


def gdn_args(**kw):
    B, H, N = kw.get("B", 1), kw.get("H", 1), kw.get("N", 64)
    base = kw.get("base", 0x10000)
    t = lambda off: _tensor(base + off, H * N * 128, N * 128, 128)
    g = lambda off: _tensor(base + off, H * N, N, 1)
    a = la.GdnPrefillArgs(B, H, N, kw.get("dk", 128), kw.get("dv", 128), la.LA_DTYPE_BF16, la.LA_DTYPE_BF16,
                          t(0), t(1 << 20), t(2 << 20), t(3 << 20), g(4 << 20), g(5 << 20), 1.0,
                          None, base + (6 << 20))
    for k, v in kw.get("set", {}).items():
        setattr(a, k, v)
    return a


def based_args(**kw):
    B, H, N = kw.get("B", 1), kw.get("H", 1), kw.get("N", 64)
    base = 0x10000
    tq = lambda off: _tensor(base + off, H * N * 16, N * 16, 16)
    tv = lambda off: _tensor(base + off, H * N * 64, N * 64, 64)
    a = la.BasedPrefillArgs(B, H, N, kw.get("df", 16), kw.get("dv", 64), la.LA_DTYPE_BF16, la.LA_DTYPE_BF16,
                            tq(0), tq(1 << 20), tv(2 << 20), tv(3 << 20), None, None,
                            base + (4 << 20), base + (5 << 20), 0.0)
    for k, v in kw.get("set", {}).items():
        setattr(a, k, v)
    return a


def call_gdn(lib, a):
    return lib.la_gdn_prefill(ctypes.byref(a), None, 0, None)


def call_based(lib, a):
    return lib.la_based_prefill(ctypes.byref(a), None, 0, None)


def test_gdn_rejections(lib):
    assert lib.la_gdn_prefill(None, None, 0, None) == la.LA_ERR_INVALID_ARGUMENT
    assert call_gdn(lib, gdn_args(dk=64, dv=64)) == la.LA_ERR_UNSUPPORTED
    assert call_gdn(lib, gdn_args(N=-1)) == la.LA_ERR_INVALID_ARGUMENT
    a = gdn_args()
    a.q = _tensor(None, 128 * 64, 128 * 64, 128)
    assert call_gdn(lib, a) == la.LA_ERR_INVALID_ARGUMENT            # null q
    a = gdn_args()
    a.k = _tensor(0x10000 + 2, 128 * 64, 128 * 64, 128)
    assert call_gdn(lib, a) == la.LA_ERR_INVALID_ARGUMENT            # misaligned base
    a = gdn_args()
    a.v = _tensor(0x10000, 128 * 64, 128 * 64, 100)
    assert call_gdn(lib, a) == la.LA_ERR_INVALID_ARGUMENT            # token stride < d and unaligned
    a = gdn_args()
    a.alpha = _tensor(0x20000, 64, 64, 2)
    assert call_gdn(lib, a) == la.LA_ERR_INVALID_ARGUMENT            # gate not contiguous along t
    a = gdn_args(set={"S_out": None})
    assert call_gdn(lib, a) == la.LA_ERR_INVALID_ARGUMENT            # missing final state
    a = gdn_args(set={"in_dtype": 7})
    assert call_gdn(lib, a) == la.LA_ERR_INVALID_ARGUMENT
    assert lib.la_gdn_prefill_workspace_size(ctypes.byref(gdn_args(dk=64, dv=64))) == 0
    # empty batch: nothing to do, no CUDA call
    assert call_gdn(lib, gdn_args(B=0)) == la.LA_OK


def test_based_rejections(lib):
    assert lib.la_based_prefill(None, None, 0, None) == la.LA_ERR_INVALID_ARGUMENT
    assert call_based(lib, based_args(df=8)) == la.LA_ERR_UNSUPPORTED
    assert call_based(lib, based_args(dv=32)) == la.LA_ERR_UNSUPPORTED
    assert call_based(lib, based_args(set={"z_out": None})) == la.LA_ERR_INVALID_ARGUMENT
    assert call_based(lib, based_args(set={"s_out": 0x10004})) == la.LA_ERR_INVALID_ARGUMENT
    assert call_based(lib, based_args(set={"decay": 0x10002})) == la.LA_ERR_INVALID_ARGUMENT  # not 4-byte aligned
    a = based_args()
    a.q = _tensor(0x10000, 16 * 64, 16 * 64, 12)
    assert call_based(lib, a) == la.LA_ERR_INVALID_ARGUMENT
    assert call_based(lib, based_args(H=0)) == la.LA_OK


def test_decode_rejections(lib):
    mk = lambda **kw: la.DecodeArgs(kw.get("variant", la.LA_VARIANT_GDN), kw.get("S", 2), 2, kw.get("dk", 128),
                                    kw.get("dv", 128), la.LA_DTYPE_BF16, la.LA_DTYPE_BF16,
                                    kw.get("q", 0x10000), 0x20000, 0x30000, kw.get("alpha", 0x40000), 0x50000,
                                    0x60000, kw.get("state", 0x70000), kw.get("z", None), 0.0, 1.0,
                                    kw.get("decay", None))
    call = lambda a: lib.la_decode_step(ctypes.byref(a), None)
    assert lib.la_decode_step(None, None) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(variant=5)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(dk=64)) == la.LA_ERR_UNSUPPORTED
    assert call(mk(variant=la.LA_VARIANT_TAYLOR)) == la.LA_ERR_UNSUPPORTED  # 128 != 16
    assert call(mk(variant=la.LA_VARIANT_TAYLOR, dk=16, dv=64)) == la.LA_ERR_INVALID_ARGUMENT  # z missing
    assert call(mk(q=None)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(alpha=None)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(state=0x70004)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(variant=la.LA_VARIANT_TAYLOR, dk=16, dv=64, z=0x80000, decay=0x90002)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(S=0)) == la.LA_OK


def test_gdn_workspace_queries_and_rejection(lib):
    rec = 16384  # records schedule: bytes of the per-chunk record (T diag(beta) and P images) of one (b,h)
    # a 4-byte ready flag per record, rounded up to 256 bytes, and the launch's scratch (an arrival
    # counter, a word per SM id up to 1024 and a progress counter, rounded up to 256 bytes)
    flags = lambda n, bh: (4 * n + 255) // 256 * 256 + 4352
    big = gdn_args(B=1, H=16, N=1 << 20)
    need_min = lib.la_gdn_prefill_workspace_size_min(ctypes.byref(big))
    need = lib.la_gdn_prefill_workspace_size(ctypes.byref(big))
    # few heads and a long sequence plan sequence segments, which need scratch
    assert need_min > 0
    assert need == 16 * (1 << 14) * rec + need_min + flags(16 * (1 << 14), 16)
    # short sequences or many heads need no segment scratch, only the records
    for B, H, N in ((4, 16, 16384), (1, 2, 64), (1, 1, 65)):
        a = gdn_args(B=B, H=H, N=N)
        assert lib.la_gdn_prefill_workspace_size_min(ctypes.byref(a)) == 0
        nrec = B * H * ((N + 63) // 64)
        assert lib.la_gdn_prefill_workspace_size(ctypes.byref(a)) == nrec * rec + flags(nrec, B * H)
    # fp32 inputs run token-serial kernels without scratch
    f32 = gdn_args(set={"in_dtype": la.LA_DTYPE_F32})
    assert lib.la_gdn_prefill_workspace_size(ctypes.byref(f32)) == 0
    assert lib.la_gdn_prefill_workspace_size_min(ctypes.byref(f32)) == 0
    # a missing, short or misaligned workspace is rejected on the host, before any launch
    assert lib.la_gdn_prefill(ctypes.byref(big), None, 0, None) == la.LA_ERR_WORKSPACE
    assert lib.la_gdn_prefill(ctypes.byref(big), ctypes.c_void_p(0x100000), need_min - 16, None) == la.LA_ERR_WORKSPACE
    assert lib.la_gdn_prefill(ctypes.byref(big), ctypes.c_void_p(0x100008), need, None) == la.LA_ERR_WORKSPACE


def test_gated_prefill_and_decode_rejections(lib):
    # the scalar gate shares the gated delta rule's arguments and validation
    call = lambda a, ws=None, n=0: lib.la_gated_prefill(ctypes.byref(a), ws, n, None)
    assert lib.la_gated_prefill(None, None, 0, None) == la.LA_ERR_INVALID_ARGUMENT
    assert call(gdn_args(dk=64, dv=64)) == la.LA_ERR_UNSUPPORTED
    assert call(gdn_args(set={"S_out": None})) == la.LA_ERR_INVALID_ARGUMENT
    a = gdn_args()
    a.alpha = _tensor(0x20000, 64, 64, 2)
    assert call(a) == la.LA_ERR_INVALID_ARGUMENT
    big = gdn_args(B=1, H=16, N=1 << 20)
    assert call(big) == la.LA_ERR_WORKSPACE
    assert call(gdn_args(B=0)) == la.LA_OK
    mk = lambda **kw: la.DecodeArgs(la.LA_VARIANT_GATED, 2, 2, kw.get("dk", 128), 128, la.LA_DTYPE_BF16,
                                    la.LA_DTYPE_BF16, 0x10000, 0x20000, 0x30000, kw.get("alpha", 0x40000), 0x50000,
                                    0x60000, 0x70000, None, 0.0, 1.0)
    assert lib.la_decode_step(ctypes.byref(mk(dk=64)), None) == la.LA_ERR_UNSUPPORTED
    assert lib.la_decode_step(ctypes.byref(mk(alpha=None)), None) == la.LA_ERR_INVALID_ARGUMENT


def test_state_op_rejections(lib):
    vp = ctypes.c_void_p
    # nothing to do: no pointer is looked at
    assert lib.la_state_rescale(None, 0, 16, None, 0.5, None) == la.LA_OK
    assert lib.la_state_gather(None, None, None, 0, 4, 16, None) == la.LA_OK
    assert lib.la_state_rescale(None, 2, 16, None, 0.5, None) == la.LA_ERR_INVALID_ARGUMENT
    assert lib.la_state_rescale(vp(0x10002), 2, 16, None, 0.5, None) == la.LA_ERR_INVALID_ARGUMENT  # misaligned
    assert lib.la_state_rescale(vp(0x10000), -1, 16, None, 0.5, None) == la.LA_ERR_INVALID_ARGUMENT
    assert lib.la_state_rescale(vp(0x10000), 1 << 30, 1 << 30, None, 0.5, None) == la.LA_ERR_INVALID_ARGUMENT
    assert lib.la_state_gather(vp(0x10000), None, vp(0x30000), 2, 2, 16, None) == la.LA_ERR_INVALID_ARGUMENT
    assert lib.la_state_gather(vp(0x10000), vp(0x20000), vp(0x30004), 2, 2, 16, None) == la.LA_ERR_INVALID_ARGUMENT
    # overlapping destination and source
    assert lib.la_state_gather(vp(0x10000), vp(0x10040), vp(0x30000), 2, 2, 16, None) == la.LA_ERR_INVALID_ARGUMENT


def test_swa_decode_rejections(lib):
    mk = lambda **kw: la.SwaDecodeArgs(kw.get("S", 2), 2, kw.get("d", 64), kw.get("window", 64), la.LA_DTYPE_BF16,
                                       la.LA_DTYPE_BF16, kw.get("q", 0x10000), 0x20000, 0x30000, 0x40000, 0x50000,
                                       kw.get("pos", 0x60000), 0x70000, 0.125)
    call = lambda a: lib.la_swa_decode_step(ctypes.byref(a), None)
    assert lib.la_swa_decode_step(None, None) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(d=60)) == la.LA_ERR_UNSUPPORTED      # not a multiple of 8
    assert call(mk(d=256)) == la.LA_ERR_UNSUPPORTED
    assert call(mk(window=0)) == la.LA_ERR_UNSUPPORTED
    assert call(mk(window=512)) == la.LA_ERR_UNSUPPORTED
    assert call(mk(q=None)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(q=0x10008)) == la.LA_ERR_INVALID_ARGUMENT  # misaligned
    assert call(mk(pos=0x60004)) == la.LA_ERR_INVALID_ARGUMENT
    assert call(mk(S=0)) == la.LA_OK


def test_notebank_rejections(lib):
    def scores(**kw):
        L, H, N, d = kw.get("L", 2), kw.get("H", 2), kw.get("N", 100), kw.get("d", 128)
        a = la.NotebankScoresArgs(L, H, N, d, la.LA_DTYPE_BF16, _tensor(0x100000, H * N * d, N * d, d),
                                  kw.get("chunk", 64), kw.get("window", 48), kw.get("d_ch", 0x200000), 0x300000,
                                  0x400000)
        return lib.la_notebank_scores(ctypes.byref(a), None)
    assert lib.la_notebank_scores(None, None) == la.LA_ERR_INVALID_ARGUMENT
    assert scores(d=48) == la.LA_ERR_UNSUPPORTED
    assert scores(d=512) == la.LA_ERR_UNSUPPORTED
    assert scores(chunk=0) == la.LA_ERR_INVALID_ARGUMENT and scores(chunk=2048) == la.LA_ERR_INVALID_ARGUMENT
    assert scores(window=0) == la.LA_ERR_INVALID_ARGUMENT
    assert scores(d_ch=0x200002) == la.LA_ERR_INVALID_ARGUMENT
    assert scores(L=0) == la.LA_OK and scores(N=0) == la.LA_OK

    def address(**kw):
        L, H, N, d = 2, 2, kw.get("N", 100), kw.get("d", 128)
        a = la.NotebankAddressArgs(L, H, N, d, kw.get("n", 3), la.LA_DTYPE_BF16, _tensor(0x100000, H * N * d, N * d, d),
                                   0x200000, 0x300000, kw.get("spans", 0x400000), 0x500000, 0x600000)
        return lib.la_notebank_address(ctypes.byref(a), None)
    assert lib.la_notebank_address(None, None) == la.LA_ERR_INVALID_ARGUMENT
    assert address(d=8) == la.LA_ERR_UNSUPPORTED
    assert address(spans=0x400004) == la.LA_ERR_INVALID_ARGUMENT
    assert address(N=0) == la.LA_ERR_INVALID_ARGUMENT
    assert address(n=0) == la.LA_OK

    def route(**kw):
        a = la.NotebankRouteArgs(kw.get("n", 10), kw.get("J", 4), kw.get("nq", 5), kw.get("R", 2), 0x100000,
                                 kw.get("u", 0x200000), None, None, 0x300000, 0x400000, 0x500000)
        return lib.la_notebank_route(ctypes.byref(a), None)
    assert lib.la_notebank_route(None, None) == la.LA_ERR_INVALID_ARGUMENT
    assert route(nq=0) == la.LA_ERR_UNSUPPORTED and route(nq=513) == la.LA_ERR_UNSUPPORTED
    assert route(R=0) == la.LA_ERR_UNSUPPORTED
    assert route(u=0x200008) == la.LA_ERR_INVALID_ARGUMENT
    assert route(J=0) == la.LA_OK


def test_cuda_error_reporting_without_a_gpu(lib):
    # nothing has failed on this thread yet; names come from the CUDA runtime's table
    assert lib.la_last_cuda_error() == 0
    assert lib.la_cuda_error_name(0) == b"cudaSuccess"
    assert lib.la_cuda_error_name(701) == b"cudaErrorLaunchOutOfResources"
