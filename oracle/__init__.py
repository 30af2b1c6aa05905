"""CPU oracle for the Gated DeltaNet mixer core (double precision).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never links, imports or calls it, and it shares no code with the CUDA library.

``gdn_oracle.c`` holds the definition (steps a1..a6 in the pages' order: causal
conv + SiLU and conv-state update, q/k L2 normalisation with the q scale, the
decay/write gates, the token-by-token delta rule, the gated RMSNorm).  This
module compiles it with gcc on first use and exposes numpy wrappers.
``chunked.py`` is a second, independent formulation (the chunked/WY form) used
only to pin the recurrence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


_LIB_F32_PATH = os.path.join(_HERE, "libgdn_oracle_f32.so")


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``libgdn_oracle.so`` next to it (gcc, OpenMP,
    double precision), and the same source with ``-DORACLE_REAL=float`` into
    ``libgdn_oracle_f32.so`` (the CPU baseline the benchmark times)."""
    with _lock:
        for path, extra in ((_LIB_PATH, []), (_LIB_F32_PATH, ["-DORACLE_REAL=float"])):
            stale = (not os.path.exists(path)) or (os.path.getmtime(path) < os.path.getmtime(_SRC))
            if force or stale:
                tmp = path + f".tmp{os.getpid()}"
                cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", *extra,
                       "-o", tmp, _SRC, "-lm"]
                subprocess.run(cmd, check=True)
                os.replace(tmp, path)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("conv_k", ctypes.c_int32), ("act", ctypes.c_int32),
                ("l2_eps", ctypes.c_double), ("rms_eps", ctypes.c_double),
                ("tiled", ctypes.c_int32), ("decay_coef", ctypes.c_int32),
                ("per_channel", ctypes.c_int32)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        lib.oracle_conv.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int, P, P, P, P, P, P]
        lib.oracle_normalize.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int, P, P, P, P]
        lib.oracle_gates.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int, P, P, P, P, P, P]
        lib.oracle_recurrence.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int] + [P] * 10
        lib.oracle_gated_norm.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int, P, P, P, P]
        lib.oracle_gdn.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int] + [P] * 20
        lib.oracle_gdn.restype = ctypes.c_int
        for f in ("oracle_conv", "oracle_normalize", "oracle_gates", "oracle_recurrence",
                  "oracle_gated_norm"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


@dataclass(frozen=True)
class Dims:
    """Geometry of one GDN layer (names follow the pages' GdnCfg / QwenConfig)."""
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    conv_k: int = 4
    act: str = "silu"          # output gate: "silu" or "sigmoid"
    l2_eps: float = 1e-6
    rms_eps: float = 1e-6
    head_map: str = "contiguous"  # key head of value head h: h // (Hv/Hk), or h % Hk ("tiled")
    decay_form: str = "A_log"     # A_log holds log A, or the decay coefficient itself ("coef")
    per_channel_decay: bool = False  # one decay per key channel: a [T, Hv, dk], dt_bias [Hv, dk]

    @property
    def conv_dim(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    def _c(self) -> _Dims:
        if self.act not in ("silu", "sigmoid"):
            raise ValueError(f"act must be 'silu' or 'sigmoid', got {self.act!r}")
        if self.head_map not in ("contiguous", "tiled") or self.decay_form not in ("A_log", "coef"):
            raise ValueError("head_map must be 'contiguous' or 'tiled', decay_form 'A_log' or 'coef'")
        return _Dims(self.n_k_heads, self.n_v_heads, self.d_k, self.d_v, self.conv_k,
                     1 if self.act == "sigmoid" else 0, self.l2_eps, self.rms_eps,
                     1 if self.head_map == "tiled" else 0, 1 if self.decay_form == "coef" else 0,
                     1 if self.per_channel_decay else 0)


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cu(cu_seqlens):
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must be a non-decreasing int vector starting at 0")
    return cu


def conv(d: Dims, cu_seqlens, x, conv_w, conv_state=None):
    """Steps a1+a2. Returns (c [T,CD] after SiLU, new conv state [N,CD,K-1])."""
    lib = _load()
    cu = _cu(cu_seqlens)
    n = cu.size - 1
    x, conv_w, cs = _f64(x), _f64(conv_w), _f64(conv_state)
    c = np.empty((int(cu[-1]), d.conv_dim))
    cs_out = np.empty((n, d.conv_dim, d.conv_k - 1))
    dd = d._c()
    lib.oracle_conv(ctypes.byref(dd), n, _ptr(cu), _ptr(x), _ptr(conv_w), _ptr(cs), _ptr(c),
                    _ptr(cs_out))
    return c, cs_out


def normalize(d: Dims, c):
    """Step a3. Returns (q_hat [T,Hk,dk] incl. the dk^-1/2 scale, k_hat, v [T,Hv,dv])."""
    lib = _load()
    c = _f64(c)
    t = c.shape[0]
    qh = np.empty((t, d.n_k_heads, d.d_k))
    kh = np.empty((t, d.n_k_heads, d.d_k))
    v = np.empty((t, d.n_v_heads, d.d_v))
    dd = d._c()
    lib.oracle_normalize(ctypes.byref(dd), t, _ptr(c), _ptr(qh), _ptr(kh), _ptr(v))
    return qh, kh, v


def gates(d: Dims, a, b, A_log, dt_bias):
    """Step a4. Returns (g, beta), each [T, Hv]; g is [T, Hv, dk] with a decay
    per key channel (then a is [T, Hv*dk] and dt_bias [Hv*dk])."""
    lib = _load()
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    t = a.shape[0]
    g = np.empty((t, d.n_v_heads, d.d_k) if d.per_channel_decay else (t, d.n_v_heads))
    beta = np.empty((t, d.n_v_heads))
    dd = d._c()
    lib.oracle_gates(ctypes.byref(dd), t, _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g),
                     _ptr(beta))
    return g, beta


def recurrence(d: Dims, cu_seqlens, q_hat, k_hat, v, g, beta, state=None, want_inter=False):
    """Step a5 (token-by-token). Returns (o [T,Hv,dv], final state [N,Hv,dk,dv], inter|None)."""
    lib = _load()
    cu = _cu(cu_seqlens)
    n = cu.size - 1
    t = int(cu[-1])
    q_hat, k_hat, v, g, beta, s0 = map(_f64, (q_hat, k_hat, v, g, beta, state))
    o = np.empty((t, d.n_v_heads, d.d_v))
    s1 = np.empty((n, d.n_v_heads, d.d_k, d.d_v))
    inter = np.empty((t, d.n_v_heads, d.d_k, d.d_v)) if want_inter else None
    dd = d._c()
    lib.oracle_recurrence(ctypes.byref(dd), n, _ptr(cu), _ptr(q_hat), _ptr(k_hat), _ptr(v),
                          _ptr(g), _ptr(beta), _ptr(s0), _ptr(s1), _ptr(inter), _ptr(o))
    return o, s1, inter


def gated_norm(d: Dims, o, z, norm_w):
    """Step a6. o, z: [T, Hv, dv] (or [T, Hv*dv]); returns y with o's shape."""
    lib = _load()
    o, z, norm_w = _f64(o), _f64(z), _f64(norm_w)
    t = o.shape[0]
    y = np.empty_like(o)
    dd = d._c()
    lib.oracle_gated_norm(ctypes.byref(dd), t, _ptr(o), _ptr(z), _ptr(norm_w), _ptr(y))
    return y


def gdn(d: Dims, cu_seqlens, x, z, a, b, conv_w, A_log, dt_bias, norm_w,
        conv_state=None, state=None, want_inter=False, want_stages=False):
    """The whole core (a1..a6) over packed sequences.

    Returns a dict with ``out`` [T, Hv*dv], ``state`` [N,Hv,dk,dv], ``conv_state``
    [N,CD,K-1], and optionally ``inter`` [T,Hv,dk,dv] and the stage outputs
    ``q_hat``, ``k_hat``, ``v``, ``g``, ``beta``.
    """
    lib = _load()
    cu = _cu(cu_seqlens)
    n = cu.size - 1
    t = int(cu[-1])
    x, z, a, b = map(_f64, (x, z, a, b))
    conv_w, A_log, dt_bias, norm_w = map(_f64, (conv_w, A_log, dt_bias, norm_w))
    cs_in, s_in = _f64(conv_state), _f64(state)
    res = {
        "out": np.empty((t, d.n_v_heads * d.d_v)),
        "state": np.empty((n, d.n_v_heads, d.d_k, d.d_v)),
        "conv_state": np.empty((n, d.conv_dim, d.conv_k - 1)),
    }
    if want_inter:
        res["inter"] = np.empty((t, d.n_v_heads, d.d_k, d.d_v))
    if want_stages:
        res["q_hat"] = np.empty((t, d.n_k_heads, d.d_k))
        res["k_hat"] = np.empty((t, d.n_k_heads, d.d_k))
        res["v"] = np.empty((t, d.n_v_heads, d.d_v))
        res["g"] = np.empty((t, d.n_v_heads, d.d_k) if d.per_channel_decay else (t, d.n_v_heads))
        res["beta"] = np.empty((t, d.n_v_heads))
    dd = d._c()
    rc = lib.oracle_gdn(ctypes.byref(dd), n, _ptr(cu), _ptr(x), _ptr(z), _ptr(a), _ptr(b),
                        _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w),
                        _ptr(cs_in), _ptr(res["conv_state"]), _ptr(s_in), _ptr(res["state"]),
                        _ptr(res.get("inter")), _ptr(res["out"]),
                        _ptr(res.get("q_hat")), _ptr(res.get("k_hat")), _ptr(res.get("v")),
                        _ptr(res.get("g")), _ptr(res.get("beta")))
    if rc != 0:
        raise MemoryError("oracle_gdn could not allocate its scratch")
    return res


_lib_f32 = None


def gdn_f32(d: Dims, cu_seqlens, x, z, a, b, conv_w, A_log, dt_bias, norm_w,
            conv_state=None, state=None):
    """The whole core (a1..a6) from the float build of the same source, for
    timing only (the CPU baseline): inputs are cast to float32, and the result
    is ``out`` [T, Hv*dv] (float32).  Parity always uses the double build."""
    global _lib_f32
    if _lib_f32 is None:
        build()
        lib = ctypes.CDLL(_LIB_F32_PATH)
        lib.oracle_gdn.argtypes = [ctypes.POINTER(_Dims), ctypes.c_int] + [ctypes.c_void_p] * 20
        lib.oracle_gdn.restype = ctypes.c_int
        _lib_f32 = lib
    cu = _cu(cu_seqlens)
    n = cu.size - 1
    t = int(cu[-1])
    f = lambda v: None if v is None else np.ascontiguousarray(np.asarray(v, dtype=np.float32))  # noqa: E731
    x, z, a, b, conv_w, A_log, dt_bias, norm_w = map(f, (x, z, a, b, conv_w, A_log, dt_bias, norm_w))
    cs_in, s_in = f(conv_state), f(state)
    out = np.empty((t, d.n_v_heads * d.d_v), dtype=np.float32)
    cs_out = np.empty((n, d.conv_dim, d.conv_k - 1), dtype=np.float32)
    s_out = np.empty((n, d.n_v_heads, d.d_k, d.d_v), dtype=np.float32)
    dd = d._c()
    rc = _lib_f32.oracle_gdn(ctypes.byref(dd), n, _ptr(cu), _ptr(x), _ptr(z), _ptr(a), _ptr(b),
                             _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(cs_in),
                             _ptr(cs_out), _ptr(s_in), _ptr(s_out), None, _ptr(out),
                             None, None, None, None, None)
    if rc != 0:
        raise MemoryError("oracle_gdn (float build) could not allocate its scratch")
    return out


def round_bf16(x):
    """Nearest bf16 value (ties to even) of each element, as float64.

    The value is first rounded to float32, as a GPU's fp32 accumulator holds it,
    then to the 8-bit bf16 mantissa."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32)).view(np.uint32)
    u = ((u.astype(np.uint64) + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def layer(d: Dims, cu_seqlens, h, w_qkv, w_z, w_a, w_b, w_out, conv_w, A_log, dt_bias,
          norm_w, conv_state=None, state=None):
    """A GDN layer's prefill around the core (qwen.rs gdn_forward: the
    in_proj_qkv / in_proj_z / in_proj_a / in_proj_b linear_multi over the hidden
    states, the core, then out_proj).  Weights are [out_features, in_features].

    Reading: the projections' results and the core's output cross the core's
    boundary in bf16, the activation type of the bf16 workloads, so they are
    rounded to bf16 here as they are on the GPU; everything else is float64.
    Returns ``gdn``'s dict plus ``h_out`` [T, hidden]."""
    h = _f64(h)
    x, z, a, b = (round_bf16(h @ _f64(w).T) for w in (w_qkv, w_z, w_a, w_b))
    res = gdn(d, cu_seqlens, x, z, a, b, conv_w, A_log, dt_bias, norm_w, conv_state=conv_state,
              state=state)
    res["h_out"] = round_bf16(res["out"]) @ _f64(w_out).T
    return res


__all__ = ["Dims", "build", "conv", "normalize", "gates", "recurrence", "gated_norm", "gdn", "gdn_f32",
           "round_bf16", "layer"]
