"""Host-side checks of the C ABI (no GPU): the library loads, exports every function
the header declares, and rejects bad arguments before touching the device."""
import ctypes

import pytest

from paged_kv_chunk_gb300 import build, capi


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def test_exports_every_header_symbol(lib):
    names = capi.header_symbols()
    assert {"oasr_paged_append", "oasr_chunk_relattn_paged", "oasr_chunk_step_paged",
            "oasr_packed_relattn_varlen", "oasr_packed_relattn_chunked", "oasr_window_commit",
            "oasr_project_qkv_pos", "oasr_status_string",
            "oasr_device_status", "oasr_selftest_wait",
            "oasr_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"


def test_status_strings(lib):
    for code in range(6):
        s = lib.oasr_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.oasr_status_string(99).decode() == "unknown status"
    assert lib.oasr_version() >= 100


FAKE = 1 << 20   # an aligned non-null pointer value that is never dereferenced


def _chunk(lib, **kw):
    a = dict(q=FAKE, kp=FAKE, vp=FAKE, nb=16, bs=16, bt=FAKE, mbps=8, cs=FAKE, u=FAKE, vb=FAKE,
             rel=FAKE, R=95, out=FAKE, B=2, T=16, H=4, D=64, scale=0.125, dt=capi.OASR_BF16)
    a.update(kw)
    return lib.oasr_chunk_relattn_paged(a["q"], a["kp"], a["vp"], a["nb"], a["bs"], a["bt"],
                                        a["mbps"], a["cs"], a["u"], a["vb"], a["rel"], a["R"],
                                        a["out"], a["B"], a["T"], a["H"], a["D"], a["scale"],
                                        a["dt"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), capi.OASR_ERR_INVALID_ARG),
    (dict(bt=None), capi.OASR_ERR_INVALID_ARG),
    (dict(B=0), capi.OASR_ERR_INVALID_ARG),
    (dict(T=-1), capi.OASR_ERR_INVALID_ARG),
    (dict(R=0), capi.OASR_ERR_INVALID_ARG),
    (dict(D=32), capi.OASR_ERR_UNSUPPORTED),
    (dict(T=65), capi.OASR_ERR_UNSUPPORTED),
    (dict(bs=24), capi.OASR_ERR_UNSUPPORTED),
    (dict(bs=4), capi.OASR_ERR_UNSUPPORTED),
    (dict(bs=512), capi.OASR_ERR_UNSUPPORTED),
    (dict(mbps=513), capi.OASR_ERR_UNSUPPORTED),   # one page past the widest table
    (dict(dt=7), capi.OASR_ERR_UNSUPPORTED),
    (dict(q=FAKE + 2), capi.OASR_ERR_INVALID_ARG),
    (dict(rel=FAKE + 8), capi.OASR_ERR_INVALID_ARG),
])
def test_chunk_rejects_bad_arguments(lib, kw, expect):
    assert _chunk(lib, **kw) == expect


def test_step_requires_chunk_pointers(lib):
    r = lib.oasr_chunk_step_paged(FAKE, None, FAKE, FAKE, FAKE, 16, 16, FAKE, 8, FAKE, FAKE, FAKE,
                                  FAKE, 95, FAKE, 2, 16, 4, 64, 0.125, capi.OASR_BF16, None)
    assert r == capi.OASR_ERR_INVALID_ARG


@pytest.mark.parametrize("args,expect", [
    (dict(D=60), capi.OASR_ERR_UNSUPPORTED),     # 120 bytes is not a multiple of 16
    (dict(k_new=None), capi.OASR_ERR_INVALID_ARG),
    (dict(nb=0), capi.OASR_ERR_INVALID_ARG),
    (dict(dt=5), capi.OASR_ERR_UNSUPPORTED),
])
def test_append_rejects_bad_arguments(lib, args, expect):
    a = dict(k_new=FAKE, v_new=FAKE, kp=FAKE, vp=FAKE, nb=16, bs=16, bt=FAKE, mbps=8, cs=FAKE, B=2,
             T=16, H=4, D=64, dt=capi.OASR_BF16)
    a.update(args)
    r = lib.oasr_paged_append(a["k_new"], a["v_new"], a["kp"], a["vp"], a["nb"], a["bs"], a["bt"],
                              a["mbps"], a["cs"], a["B"], a["T"], a["H"], a["D"], a["dt"], None)
    assert r == expect


@pytest.mark.parametrize("args,expect", [
    (dict(ns=1025), capi.OASR_ERR_UNSUPPORTED),
    (dict(D=128), capi.OASR_ERR_UNSUPPORTED),
    (dict(total=0), capi.OASR_ERR_INVALID_ARG),
    (dict(cu=None), capi.OASR_ERR_INVALID_ARG),
    (dict(k=FAKE + 4), capi.OASR_ERR_INVALID_ARG),
])
def test_packed_rejects_bad_arguments(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu=FAKE, ns=4, maxlen=100, total=300, u=FAKE, vb=FAKE,
             rel=FAKE, R=199, out=FAKE, H=8, D=64, dt=capi.OASR_BF16)
    a.update(args)
    r = lib.oasr_packed_relattn_varlen(a["q"], a["k"], a["v"], a["cu"], a["ns"], a["maxlen"],
                                       a["total"], a["u"], a["vb"], a["rel"], a["R"], a["out"],
                                       a["H"], a["D"], 0.125, a["dt"], None)
    assert r == expect


@pytest.mark.parametrize("args,expect", [
    (dict(cs=0), capi.OASR_ERR_INVALID_ARG),
    (dict(left=-1), capi.OASR_ERR_INVALID_ARG),
    (dict(ns=1025), capi.OASR_ERR_UNSUPPORTED),
    (dict(D=128), capi.OASR_ERR_UNSUPPORTED),
    (dict(total=0), capi.OASR_ERR_INVALID_ARG),
    (dict(cu=None), capi.OASR_ERR_INVALID_ARG),
    (dict(k=FAKE + 4), capi.OASR_ERR_INVALID_ARG),
])
def test_chunked_rejects_bad_arguments(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, cu=FAKE, ns=4, maxlen=100, total=300, u=FAKE, vb=FAKE,
             rel=FAKE, R=199, out=FAKE, H=8, D=64, cs=8, left=7, dt=capi.OASR_BF16)
    a.update(args)
    r = lib.oasr_packed_relattn_chunked(a["q"], a["k"], a["v"], a["cu"], a["ns"], a["maxlen"],
                                        a["total"], a["u"], a["vb"], a["rel"], a["R"], a["out"],
                                        a["H"], a["D"], 0.125, a["cs"], a["left"], a["dt"], None)
    assert r == expect


@pytest.mark.parametrize("args,expect", [
    (dict(bt=None), capi.OASR_ERR_INVALID_ARG),
    (dict(cs=None), capi.OASR_ERR_INVALID_ARG),
    (dict(B=0), capi.OASR_ERR_INVALID_ARG),
    (dict(bs=0), capi.OASR_ERR_INVALID_ARG),
    (dict(T=-1), capi.OASR_ERR_INVALID_ARG),
    (dict(window=-1), capi.OASR_ERR_INVALID_ARG),
    (dict(mbps=513), capi.OASR_ERR_UNSUPPORTED),
])
def test_window_commit_rejects_bad_arguments(lib, args, expect):
    a = dict(bt=FAKE, cs=FAKE, B=4, mbps=8, bs=16, T=16, window=64)
    a.update(args)
    assert lib.oasr_window_commit(a["bt"], a["cs"], a["B"], a["mbps"], a["bs"], a["T"], a["window"],
                                  None) == expect


@pytest.mark.parametrize("args,expect", [
    (dict(x=None), capi.OASR_ERR_INVALID_ARG),
    (dict(M=0), capi.OASR_ERR_INVALID_ARG),
    (dict(dm=192, H=3), capi.OASR_ERR_UNSUPPORTED),     # not a multiple of 128
    (dict(dm=256, H=2), capi.OASR_ERR_UNSUPPORTED),     # d_model != 64 H
    (dict(dt=capi.OASR_F32), capi.OASR_ERR_UNSUPPORTED),
    (dict(q=FAKE + 4), capi.OASR_ERR_INVALID_ARG),
])
def test_projection_rejects_bad_arguments(lib, args, expect):
    a = dict(x=FAKE, q=FAKE, M=1024, R=287, dm=256, H=4, dt=capi.OASR_BF16)
    a.update(args)
    r = lib.oasr_project_qkv_pos(a["x"], FAKE, FAKE, FAKE, FAKE, a["q"], FAKE, FAKE, FAKE, a["M"],
                                 a["R"], a["dm"], a["H"], a["dt"], None)
    assert r == expect


def test_device_status_needs_pointer(lib):
    assert lib.oasr_device_status(ctypes.cast(None, ctypes.POINTER(ctypes.c_uint)), 0) == \
        capi.OASR_ERR_INVALID_ARG


def test_binding_raises_on_cpu_tensors():
    import torch
    x = torch.zeros(2, 16, 4, 64)
    with pytest.raises(ValueError):
        capi.oasr_paged_append(x, x, torch.zeros(16, 16, 4, 64), torch.zeros(16, 16, 4, 64),
                               torch.zeros(2, 8, dtype=torch.int32),
                               torch.zeros(2, dtype=torch.int32))


def test_binding_checks_shapes_before_any_pointer():
    """Sizes the kernels derive from one tensor must hold for the others: a V pool or an
    output smaller than its partner is refused before anything reaches the library."""
    import torch
    bf = torch.bfloat16
    q = torch.zeros(2, 16, 4, 64, dtype=bf)
    kp, vp_small = torch.zeros(16, 16, 4, 64, dtype=bf), torch.zeros(8, 16, 4, 64, dtype=bf)
    bt, cs = torch.zeros(2, 8, dtype=torch.int32), torch.zeros(2, dtype=torch.int32)
    uv, rel = torch.zeros(4, 64, dtype=bf), torch.zeros(47, 4, 64, dtype=bf)
    for call in (lambda: capi.oasr_chunk_relattn_paged(q, kp, vp_small, bt, cs, uv, uv, rel),
                 lambda: capi.oasr_chunk_step_paged(q, q, q, kp, vp_small, bt, cs, uv, uv, rel)):
        with pytest.raises(ValueError, match="v_pool"):
            call()
    x, w, bqkv = torch.zeros(32, 256, dtype=bf), torch.zeros(768, 256, dtype=bf), torch.zeros(768, dtype=bf)
    pe, wp = torch.zeros(47, 256, dtype=bf), torch.zeros(256, 256, dtype=bf)
    with pytest.raises(ValueError, match="q, k, v must be"):
        capi.oasr_project_qkv_pos(x, w, bqkv, pe, wp, 4, q=torch.zeros(16, 4, 64, dtype=bf))
    with pytest.raises(ValueError, match="q, k, v must be"):
        capi.oasr_project_qkv_pos(x, w, bqkv, pe, wp, 4, rel=torch.zeros(46, 4, 64, dtype=bf))


@pytest.mark.parametrize("limit_us", [0, 2000001])
def test_selftest_wait_rejects_bad_limits(lib, limit_us):
    assert lib.oasr_selftest_wait(limit_us, None) == capi.OASR_ERR_INVALID_ARG


@pytest.mark.parametrize("flag", ["1", ""])
def test_nvtx_ranges_are_opt_in(flag):
    """With OASR_NVTX=1 every library call of the binding is wrapped in an NVTX range;
    otherwise the binding's functions are the plain ones."""
    import os
    import subprocess
    import sys
    code = ("from paged_kv_chunk_gb300 import capi\n"
            "names = ['oasr_paged_append', 'oasr_chunk_relattn_paged', 'oasr_chunk_step_paged',"
            " 'oasr_packed_relattn_varlen', 'oasr_packed_relattn_chunked', 'oasr_window_commit',"
            " 'oasr_project_qkv_pos', 'oasr_selftest_wait']\n"
            "print(sum(hasattr(getattr(capi, n), '__wrapped__') for n in names))\n")
    env = dict(os.environ, OASR_NVTX=flag)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, check=True,
                         capture_output=True, text=True).stdout.split()
    assert int(out[-1]) == (8 if flag == "1" else 0)
