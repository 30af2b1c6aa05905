"""Host-side failure injection (GDN_FAULT) and the timeout status, on the CPU.

The pages' engine fails closed and tests that path with a test-only fail point
(cortiq-engine 0.8.76 pipeline.rs, nll_test_fail_at; graph_failed ->
clear_sequence_state).  Here a call whose site GDN_FAULT lists validates its
arguments and returns GDN_ERR_INJECTED before it enqueues anything.  The calls
below get host buffers filled with a sentinel: an injected call returns before
any CUDA call, so the buffers must come back untouched (no GPU is needed).
"""
import ctypes

import numpy as np
import pytest

import gated_deltanet_linear_mixer_gb300 as gdn
from gated_deltanet_linear_mixer_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gdn.load()


def _dims(**kw):
    base = dict(n_k_heads=2, n_v_heads=4, d_k=32, d_v=32, conv_k=4, dtype=0, act=0,
                l2_eps=1e-6, rms_eps=1e-6)
    base.update(kw)
    return gdn._Dims(**base)


class Buffers:
    """Aligned host buffers standing in for every pointer argument, each filled
    with a sentinel so that any write would show."""

    def __init__(self):
        self.arrays = []

    def get(self, n=4096):
        a = np.full(n + 16, 12345.0, dtype=np.float32)
        off = (-a.ctypes.data % 16) // 4
        view = a[off:off + n]
        self.arrays.append(view)
        return ctypes.c_void_p(view.ctypes.data)

    def untouched(self):
        return all(np.all(v == 12345.0) for v in self.arrays)


def _params(buf):
    return gdn._Params(buf.get().value, buf.get().value, buf.get().value, buf.get().value)


SITES = {
    "prefill": lambda lib, d, p, b, cu: lib.gdn_prefill(
        ctypes.byref(d), ctypes.byref(p), 1, b.get(), cu, b.get(), b.get(), b.get(), b.get(),
        b.get(), b.get(), b.get(), b.get(), b.get(), b.get(), 1 << 20, None),
    "conv": lambda lib, d, p, b, cu: lib.gdn_conv(
        ctypes.byref(d), ctypes.byref(p), 1, b.get(), cu, b.get(), b.get(), b.get(), b.get(),
        b.get(), b.get(), b.get(), b.get(), None),
    "decode": lambda lib, d, p, b, cu: lib.gdn_decode(
        ctypes.byref(d), ctypes.byref(p), 2, 1, b.get(), b.get(), b.get(), b.get(), b.get(),
        b.get(), None, b.get(), None),
    "verify": lambda lib, d, p, b, cu: lib.gdn_verify(
        ctypes.byref(d), ctypes.byref(p), 2, 3, b.get(), b.get(), b.get(), b.get(), b.get(),
        b.get(), b.get(), None),
    "commit": lambda lib, d, p, b, cu: lib.gdn_decode_commit(
        ctypes.byref(d), 2, 3, b.get(), b.get(), b.get(), b.get(), b.get(), None),
}


@pytest.mark.parametrize("site", sorted(SITES))
@pytest.mark.parametrize("listed", ["{site}", "all", "decode_x,{site}", "{site},layer"])
def test_listed_site_fails_before_any_work(lib, monkeypatch, site, listed):
    monkeypatch.setenv("GDN_FAULT", listed.format(site=site))
    buf = Buffers()
    cu = (ctypes.c_int32 * 2)(0, 4)
    st = SITES[site](lib, _dims(), _params(buf), buf, ctypes.cast(cu, ctypes.c_void_p))
    assert st == gdn.GDN_ERR_INJECTED, (st, lib.gdn_last_error())
    msg = lib.gdn_last_error().decode()
    assert "fault injected" in msg and "nothing was enqueued" in msg
    assert buf.untouched()


def test_validation_comes_before_injection(lib, monkeypatch):
    """A call with a bad argument reports that argument, injected or not: the
    injection point sits after validation."""
    monkeypatch.setenv("GDN_FAULT", "all")
    buf = Buffers()
    cu = (ctypes.c_int32 * 2)(0, 4)
    st = SITES["prefill"](lib, _dims(d_k=48), _params(buf), buf, ctypes.cast(cu, ctypes.c_void_p))
    assert st == 2 and "d_k and d_v" in lib.gdn_last_error().decode()


def test_layer_site(lib, monkeypatch):
    monkeypatch.setenv("GDN_FAULT", "layer")
    buf = Buffers()
    d = _dims(dtype=1)
    cu = (ctypes.c_int32 * 2)(0, 4)
    proj = gdn._Proj(*(buf.get().value for _ in range(5)))
    need = ctypes.c_size_t(0)
    assert lib.gdn_layer_prefill_workspace_size(ctypes.byref(d), 64, 1, ctypes.cast(cu, ctypes.c_void_p),
                                                ctypes.byref(need)) == 0
    ws = np.zeros(need.value // 4 + 256, dtype=np.float32)
    ws_ptr = ctypes.c_void_p(ws.ctypes.data + (-ws.ctypes.data % 256))
    st = lib.gdn_layer_prefill(ctypes.byref(d), ctypes.byref(_params(buf)), ctypes.byref(proj), 64, 1,
                               buf.get(), ctypes.cast(cu, ctypes.c_void_p), buf.get(), None, None,
                               None, None, buf.get(), ws_ptr, need.value, None)
    assert st == gdn.GDN_ERR_INJECTED
    assert buf.untouched() and not ws.any()


def test_unlisted_site_is_not_injected(lib, monkeypatch):
    """An unrelated site leaves the call alone: here validation then refuses a
    missing workspace, before any launch."""
    monkeypatch.setenv("GDN_FAULT", "decode,verify")
    buf = Buffers()
    d = _dims(dtype=1, d_k=128, d_v=128)
    cu = (ctypes.c_int32 * 2)(0, 200)
    p = _params(buf)
    st = lib.gdn_prefill(ctypes.byref(d), ctypes.byref(p), 1, buf.get(), ctypes.cast(cu, ctypes.c_void_p),
                         buf.get(), buf.get(), buf.get(), buf.get(), None, None, None, None,
                         buf.get(), None, 0, None)
    assert st == 4, lib.gdn_last_error()  # GDN_ERR_WORKSPACE: not injected


def test_status_names_cover_the_header():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "gdn.h")).read()
    declared = {int(v): k for k, v in re.findall(r"(GDN_\w+) = (\d+)", text.split("} gdn_status;")[0])}
    assert declared == gdn.STATUS_NAMES
