"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every
symbol include/gdn.h declares, and rejects bad arguments on the host (these
calls fail validation before any CUDA call, so no GPU is needed)."""
import ctypes
import os
import re
import threading

import pytest

import gated_deltanet_linear_mixer_gb300 as gdn
from gated_deltanet_linear_mixer_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gdn.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return set(re.findall(r"^(?:gdn_status|const char\*|size_t)\s+(gdn_\w+)\(", text, re.M))


def test_header_declares_the_exports():
    assert _declared() == set(gdn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert "sm_103a" in gdn.version()


def _dims(**kw):
    base = dict(n_k_heads=16, n_v_heads=32, d_k=128, d_v=128, conv_k=4, dtype=1, act=0,
                l2_eps=1e-6, rms_eps=1e-6)
    base.update(kw)
    return gdn._Dims(**base)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
PARAMS = gdn._Params(0x10000, 0x10000, 0x10000, 0x10000)


def _prefill(lib, d, n_seq=1, cu_host=(0, 4), x=FAKE, ws=None, ws_bytes=0):
    cu = (ctypes.c_int32 * len(cu_host))(*cu_host)
    return lib.gdn_prefill(ctypes.byref(d), ctypes.byref(PARAMS), n_seq, FAKE,
                           ctypes.cast(cu, ctypes.c_void_p), x, FAKE, FAKE, FAKE, None, None,
                           None, None, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(d_k=48), 2, "d_k and d_v"),
    (dict(d_v=256), 2, "d_k and d_v"),
    (dict(n_v_heads=24, n_k_heads=16), 2, "multiple of n_k_heads"),
    (dict(conv_k=5), 2, "conv_k"),
    (dict(conv_k=1), 2, "conv_k"),
    (dict(dtype=7), 1, "dtype"),
    (dict(act=3), 1, "act"),
    (dict(rms_eps=0.0), 1, "eps"),
    (dict(n_k_heads=0), 1, "head counts"),
])
def test_bad_dims_are_rejected(lib, kw, status, msg):
    assert _prefill(lib, _dims(**kw)) == status
    assert msg in lib.gdn_last_error().decode()


def test_bad_cu_seqlens_are_rejected(lib):
    assert _prefill(lib, _dims(), 1, (1, 4)) == 1
    assert "cu_seqlens[0]" in lib.gdn_last_error().decode()
    assert _prefill(lib, _dims(), 2, (0, 4, 3)) == 1
    assert "decreases" in lib.gdn_last_error().decode()
    assert _prefill(lib, _dims(), -1, (0,)) == 1


def test_misaligned_pointer_is_rejected(lib):
    assert _prefill(lib, _dims(), x=ctypes.c_void_p(0x10002)) == 1
    assert "aligned" in lib.gdn_last_error().decode()


def test_null_params_rejected(lib):
    d = _dims()
    cu = (ctypes.c_int32 * 2)(0, 4)
    st = lib.gdn_prefill(ctypes.byref(d), None, 1, FAKE, ctypes.cast(cu, ctypes.c_void_p),
                         FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, None, 0, None)
    assert st == 1 and "params" in lib.gdn_last_error().decode()
    assert lib.gdn_prefill(None, ctypes.byref(PARAMS), 1, FAKE, ctypes.cast(cu, ctypes.c_void_p),
                           FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, None, 0, None) == 1


@pytest.mark.parametrize("T", [0, 17, -3])
def test_decode_token_count_is_checked(lib, T):
    d = _dims()
    st = lib.gdn_decode(ctypes.byref(d), ctypes.byref(PARAMS), 4, T, FAKE, FAKE, FAKE, FAKE,
                        FAKE, None, None, FAKE, None)
    assert st == 1 and "T must be" in lib.gdn_last_error().decode()


def test_empty_calls_are_no_ops(lib):
    d = _dims()
    assert lib.gdn_decode(ctypes.byref(d), ctypes.byref(PARAMS), 0, 1, None, None, None, None,
                          None, None, None, None, None) == 0
    assert _prefill(lib, d, 0, (0,), x=None) == 0


def test_workspace_query(lib):
    d = _dims()
    cu = (ctypes.c_int32 * 3)(0, 4096, 5000)
    n = ctypes.c_size_t(123)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(d), 2, ctypes.cast(cu, ctypes.c_void_p),
                                          ctypes.byref(n)) == 0
    assert n.value % 256 == 0


def test_last_error_is_per_thread(lib):
    assert _prefill(lib, _dims(d_k=48)) == 2
    seen = {}

    def other():
        seen["msg"] = lib.gdn_last_error().decode()

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen["msg"] == ""
    assert "d_k" in lib.gdn_last_error().decode()


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        gdn.load(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("kw,msg", [
    (dict(head_map=2), "head_map"),
    (dict(decay_form=-1), "decay_form"),
    (dict(decay_per_channel=2), "decay_per_channel"),
])
def test_bad_options_are_rejected(lib, kw, msg):
    assert _prefill(lib, _dims(**kw)) == 1
    assert msg in lib.gdn_last_error().decode()


@pytest.mark.parametrize("T", [0, 17])
def test_verify_token_count_is_checked(lib, T):
    d = _dims()
    st = lib.gdn_verify(ctypes.byref(d), ctypes.byref(PARAMS), 4, T, FAKE, FAKE, FAKE, FAKE,
                        FAKE, None, FAKE, None)
    assert st == 1 and "T must be" in lib.gdn_last_error().decode()


def test_verify_pointer_checks(lib):
    d = _dims()
    assert lib.gdn_verify(ctypes.byref(d), ctypes.byref(PARAMS), 0, 4, None, None, None, None,
                          None, None, None, None) == 0
    assert lib.gdn_verify(ctypes.byref(d), ctypes.byref(PARAMS), 2, 4, FAKE, FAKE, FAKE, FAKE,
                          None, None, FAKE, None) == 1
    assert "NULL" in lib.gdn_last_error().decode()
    assert lib.gdn_verify(ctypes.byref(d), ctypes.byref(PARAMS), 2, 4, FAKE, FAKE, FAKE, FAKE,
                          ctypes.c_void_p(0x10008), None, FAKE, None) == 1
    assert "aligned" in lib.gdn_last_error().decode()


def _proj(addr=0x10000):
    p = ctypes.c_void_p(addr)
    return gdn._Proj(p, p, p, p, p)


def _layer(lib, d, proj, hidden=64, n_seq=1, cu_host=(0, 4), ws=None, ws_bytes=0):
    cu = (ctypes.c_int32 * len(cu_host))(*cu_host)
    return lib.gdn_layer_prefill(ctypes.byref(d), ctypes.byref(PARAMS),
                                 ctypes.byref(proj) if proj is not None else None, hidden, n_seq,
                                 FAKE, ctypes.cast(cu, ctypes.c_void_p), FAKE, None, None, None,
                                 None, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("hidden", [0, 7, 12, -8])
def test_layer_hidden_is_checked(lib, hidden):
    d = _dims()
    cu = (ctypes.c_int32 * 2)(0, 4)
    n = ctypes.c_size_t(0)
    assert lib.gdn_layer_prefill_workspace_size(ctypes.byref(d), hidden, 1,
                                                ctypes.cast(cu, ctypes.c_void_p),
                                                ctypes.byref(n)) == 1
    assert "hidden" in lib.gdn_last_error().decode()


def test_layer_workspace_covers_the_core(lib):
    d = _dims()
    cu = (ctypes.c_int32 * 3)(0, 4096, 5000)
    core, layer = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(d), 2, ctypes.cast(cu, ctypes.c_void_p),
                                          ctypes.byref(core)) == 0
    assert lib.gdn_layer_prefill_workspace_size(ctypes.byref(d), 2048, 2,
                                                ctypes.cast(cu, ctypes.c_void_p),
                                                ctypes.byref(layer)) == 0
    # x, z, a, b and y (bf16) plus the core's own workspace, all inside the layer's
    cd = 2 * 16 * 128 + 32 * 128
    act = 5000 * (cd + 2 * 32 * 128 + 2 * 32) * 2
    assert layer.value >= core.value + act and layer.value % 256 == 0


def test_layer_refusals(lib):
    assert _layer(lib, _dims(dtype=0), _proj()) == 2
    assert "bf16" in lib.gdn_last_error().decode()
    assert _layer(lib, _dims(decay_per_channel=1), _proj()) == 2
    assert "per-channel" in lib.gdn_last_error().decode()
    assert _layer(lib, _dims(), None) == 1
    assert "projection" in lib.gdn_last_error().decode()
    assert _layer(lib, _dims(), _proj(0x10004)) == 1
    assert "aligned" in lib.gdn_last_error().decode()
    # no sequences: nothing to do
    assert _layer(lib, _dims(), _proj(), n_seq=0, cu_host=(0,)) == 0
    # too small a workspace is refused before any launch
    assert _layer(lib, _dims(), _proj(), ws=FAKE, ws_bytes=256) == 4
    assert "workspace" in lib.gdn_last_error().decode()


def test_sequence_count_limit(lib):
    """More than GDN_MAX_SEQUENCES sequences is refused on the host."""
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    limit = int(re.search(r"#define GDN_MAX_SEQUENCES (\d+)", text).group(1))
    d = _dims()
    for fn in ("gdn_decode", "gdn_verify"):
        if fn == "gdn_decode":
            args = [ctypes.byref(d), ctypes.byref(PARAMS), limit + 1, 1, FAKE, FAKE, FAKE, FAKE,
                    FAKE, None, None, FAKE, None]
        else:
            args = [ctypes.byref(d), ctypes.byref(PARAMS), limit + 1, 1, FAKE, FAKE, FAKE, FAKE,
                    FAKE, None, FAKE, None]
        assert getattr(lib, fn)(*args) == 1
        assert "GDN_MAX_SEQUENCES" in lib.gdn_last_error().decode()
    assert lib.gdn_decode_commit(ctypes.byref(d), limit + 1, 1, FAKE, FAKE, FAKE, FAKE, None,
                                 None) == 1
    cu = (ctypes.c_int32 * (limit + 2))(*range(limit + 2))
    n = ctypes.c_size_t(0)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(d), limit + 1,
                                          ctypes.cast(cu, ctypes.c_void_p), ctypes.byref(n)) == 2
    assert "GDN_MAX_SEQUENCES" in lib.gdn_last_error().decode()


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/gdn.h compiles as strict C99, and a C program that takes the
    address of every declared entry point links against libgdn.so."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    names = sorted(_declared())
    src = tmp_path / "use_gdn.c"
    src.write_text('#include "gdn.h"\n#include <stdio.h>\n'
                   "typedef void (*fp)(void);\n"
                   "int main(void) {\n"
                   "    fp table[] = {\n" +
                   "".join(f"        (fp){n},\n" for n in names) +
                   "    };\n"
                   '    printf("%d %s\\n", (int)(sizeof table / sizeof table[0]), gdn_version());\n'
                   "    return 0;\n}\n")
    exe = tmp_path / "use_gdn"
    libdir = os.path.dirname(gdn.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o",
                        str(exe), "-L", libdir, "-lgdn", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split()[0] == str(len(names))
