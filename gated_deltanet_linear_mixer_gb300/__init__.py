"""Gated DeltaNet mixer core for GB300 (sm_103a): Python binding of libgdn.so.

The binding only marshals arguments: it checks tensor shapes/dtypes/devices,
takes raw device pointers and the current CUDA stream, and calls the C ABI
declared in ``include/gdn.h``.  Every step of the computation runs in the CUDA
kernels of ``libgdn.so``; there is no CPU or PyTorch fallback.  If the library
is missing the calls raise.  Build it with ``gated_deltanet_linear_mixer_gb300._build.build()``
(or ``__graft_entry__.build()``).

Entry points (same names as the C ABI, without the ``gdn_`` prefix):
``conv``, ``prefill``, ``prefill_workspace_size``, ``decode``, ``decode_commit``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_CUDA", 4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_TIMEOUT",
                6: "GDN_ERR_INJECTED"}
GDN_ERR_TIMEOUT, GDN_ERR_INJECTED = 5, 6
DTYPE_F32, DTYPE_BF16 = 0, 1
ACT_SILU, ACT_SIGMOID = 0, 1

# Every symbol include/gdn.h declares.
EXPORTS = ("gdn_conv", "gdn_prefill_workspace_size", "gdn_prefill", "gdn_prefill_noalloc",
           "gdn_prefill_noalloc_scratch_bytes", "gdn_decode", "gdn_verify", "gdn_decode_commit",
           "gdn_layer_prefill_workspace_size", "gdn_layer_prefill",
           "gdn_timing_enable", "gdn_timing_report", "gdn_device_error", "gdn_sync_status",
           "gdn_last_error", "gdn_version")


class GDNError(RuntimeError):
    """A libgdn call returned a status other than GDN_OK."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Dims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("conv_k", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("l2_eps", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("head_map", ctypes.c_int32), ("decay_form", ctypes.c_int32),
                ("decay_per_channel", ctypes.c_int32)]


class _Params(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p)]


class _Proj(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_z", ctypes.c_void_p), ("w_a", ctypes.c_void_p),
                ("w_b", ctypes.c_void_p), ("w_out", ctypes.c_void_p)]


_lib = None


def load(path: str | None = None):
    """Load libgdn.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libgdn.so not found at {path}; build it first "
                           "(gated_deltanet_linear_mixer_gb300._build.build())")
    lib = ctypes.CDLL(path)
    P, I32, PD = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(_Dims)
    PP = ctypes.POINTER(_Params)
    lib.gdn_conv.argtypes = [PD, PP, I32, P, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_prefill_workspace_size.argtypes = [PD, I32, P, ctypes.POINTER(ctypes.c_size_t)]
    lib.gdn_prefill.argtypes = [PD, PP, I32, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.gdn_prefill_noalloc.argtypes = [PD, PP, I32, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_prefill_noalloc_scratch_bytes.argtypes = []
    lib.gdn_prefill_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.gdn_decode.argtypes = [PD, PP, I32, I32, P, P, P, P, P, P, P, P, P]
    lib.gdn_verify.argtypes = [PD, PP, I32, I32, P, P, P, P, P, P, P, P]
    lib.gdn_decode_commit.argtypes = [PD, I32, I32, P, P, P, P, P, P]
    lib.gdn_layer_prefill_workspace_size.argtypes = [PD, I32, I32, P, ctypes.POINTER(ctypes.c_size_t)]
    lib.gdn_layer_prefill.argtypes = [PD, PP, ctypes.POINTER(_Proj), I32, I32, P, P, P, P, P, P, P,
                                      P, P, ctypes.c_size_t, P]
    for f in ("gdn_conv", "gdn_prefill_workspace_size", "gdn_prefill", "gdn_prefill_noalloc",
              "gdn_decode", "gdn_verify", "gdn_decode_commit", "gdn_layer_prefill_workspace_size",
              "gdn_layer_prefill"):
        getattr(lib, f).restype = ctypes.c_int
    lib.gdn_timing_enable.argtypes = [I32]
    lib.gdn_timing_enable.restype = ctypes.c_int
    lib.gdn_timing_report.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
    lib.gdn_timing_report.restype = ctypes.c_size_t
    lib.gdn_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), I32]
    lib.gdn_device_error.restype = ctypes.c_int
    lib.gdn_sync_status.argtypes = [P]
    lib.gdn_sync_status.restype = ctypes.c_int
    lib.gdn_last_error.restype = ctypes.c_char_p
    lib.gdn_last_error.argtypes = []
    lib.gdn_version.restype = ctypes.c_char_p
    lib.gdn_version.argtypes = []
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != GDN_OK:
        raise GDNError(fn, status, load().gdn_last_error().decode(errors="replace"))


@dataclass(frozen=True)
class Dims:
    """Geometry of one GDN layer: Hk, Hv, d_k, d_v, K, activation dtype, gate act."""
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    conv_k: int = 4
    dtype: torch.dtype = torch.bfloat16
    act: str = "silu"
    l2_eps: float = 1e-6
    rms_eps: float = 1e-6
    head_map: str = "contiguous"   # value head h reads key head h // (Hv/Hk), or h % Hk ("tiled")
    decay_form: str = "A_log"      # Params.A_log holds log A, or the decay coefficient ("coef")
    per_channel_decay: bool = False  # one decay per key channel: a [T, Hv*dk], dt_bias [Hv*dk]

    @property
    def conv_dim(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def gate_width(self) -> int:
        """Columns of the decay-gate input a (and entries of dt_bias)."""
        return self.n_v_heads * (self.d_k if self.per_channel_decay else 1)

    def c(self) -> _Dims:
        if self.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("activation dtype must be torch.float32 or torch.bfloat16")
        if self.act not in ("silu", "sigmoid"):
            raise ValueError("act must be 'silu' or 'sigmoid'")
        if self.head_map not in ("contiguous", "tiled"):
            raise ValueError("head_map must be 'contiguous' or 'tiled'")
        if self.decay_form not in ("A_log", "coef"):
            raise ValueError("decay_form must be 'A_log' or 'coef'")
        return _Dims(self.n_k_heads, self.n_v_heads, self.d_k, self.d_v, self.conv_k,
                     DTYPE_BF16 if self.dtype == torch.bfloat16 else DTYPE_F32,
                     ACT_SIGMOID if self.act == "sigmoid" else ACT_SILU,
                     self.l2_eps, self.rms_eps, 1 if self.head_map == "tiled" else 0,
                     1 if self.decay_form == "coef" else 0, 1 if self.per_channel_decay else 0)


@dataclass
class Params:
    """Per-layer fp32 parameters on the GPU: conv_w [CD,K], A_log [Hv], dt_bias [Hv], norm_w [dv]."""
    conv_w: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    norm_w: torch.Tensor

    def c(self, d: Dims) -> _Params:
        _t(self.conv_w, "conv_w", torch.float32, (d.conv_dim, d.conv_k))
        _t(self.A_log, "A_log", torch.float32, (d.n_v_heads,))
        _t(self.dt_bias, "dt_bias", torch.float32, (d.gate_width,))
        _t(self.norm_w, "norm_w", torch.float32, (d.d_v,))
        return _Params(self.conv_w.data_ptr(), self.A_log.data_ptr(), self.dt_bias.data_ptr(),
                       self.norm_w.data_ptr())


def _t(x, name, dtype, shape=None, cuda=True):
    if x is None:
        return None
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda and not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return x


def _p(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cu_pair(cu_seqlens, device):
    """cu_seqlens as (device int32 tensor, host int32 tensor).

    Accepts a list, a tensor (host or device), or a ready (device, host) pair,
    which avoids a device-to-host copy per call."""
    if isinstance(cu_seqlens, tuple) and len(cu_seqlens) == 2:
        dev, host = cu_seqlens
        _t(dev, "cu_seqlens (device)", torch.int32)
        _t(host, "cu_seqlens (host)", torch.int32, cuda=False)
        if host.is_cuda or host.numel() != dev.numel():
            raise ValueError("cu_seqlens pair must be (device tensor, host tensor) of equal size")
        return dev, host
    if isinstance(cu_seqlens, torch.Tensor):
        host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
        dev = cu_seqlens if (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32
                             and cu_seqlens.is_contiguous()) else host.to(device)
    else:
        host = torch.tensor(list(cu_seqlens), dtype=torch.int32)
        dev = host.to(device)
    return dev, host


def version() -> str:
    return load().gdn_version().decode()


def timing_enable(on: bool = True) -> None:
    """Start (clearing totals) or stop per-kernel CUDA-event timing in libgdn."""
    _check("gdn_timing_enable", load().gdn_timing_enable(1 if on else 0))


def timing_report() -> dict:
    """{kernel name: (launches, total ms)} recorded since timing_enable(True)."""
    lib = load()
    need = lib.gdn_timing_report(None, 0)
    buf = ctypes.create_string_buffer(max(need, 1))
    lib.gdn_timing_report(buf, len(buf))
    rep = {}
    for line in buf.value.decode().splitlines():
        name, n, ms = line.split()
        rep[name] = (int(n), float(ms))
    return rep


def device_error(reset: bool = True) -> int:
    """The sticky device-side error word (0 = none); waits for the device."""
    code = ctypes.c_int32(0)
    _check("gdn_device_error", load().gdn_device_error(ctypes.byref(code), 1 if reset else 0))
    return int(code.value)


def sync_status(device=None) -> None:
    """gdn_sync_status on the current stream: waits for it, then raises GDNError
    (status GDN_ERR_TIMEOUT) if a bounded device wait gave up since the last
    check; the word is cleared either way."""
    _check("gdn_sync_status", load().gdn_sync_status(_stream(device)))


def conv(d: Dims, params: Params, cu_seqlens, x, a, b, conv_state_in=None, conv_state_out=None,
         qkv_out=None, g_out=None, beta_out=None):
    """gdn_conv: prologue only.  Returns (qkv_out [T,CD], g [T,Hv], beta [T,Hv])."""
    lib = load()
    dev = x.device
    cu_d, cu_h = _cu_pair(cu_seqlens, dev)
    n = cu_h.numel() - 1
    t = int(cu_h[-1]) if n > 0 else 0
    _t(x, "x", d.dtype, (t, d.conv_dim))
    _t(a, "a", d.dtype, (t, d.gate_width))
    _t(b, "b", d.dtype, (t, d.n_v_heads))
    cs_shape = (n, d.conv_dim, d.conv_k - 1)
    _t(conv_state_in, "conv_state_in", d.dtype, cs_shape)
    _t(conv_state_out, "conv_state_out", d.dtype, cs_shape)
    qkv_out = qkv_out if qkv_out is not None else torch.empty_like(x)
    g_out = g_out if g_out is not None else torch.empty((t, d.n_v_heads), device=dev)
    beta_out = beta_out if beta_out is not None else torch.empty((t, d.n_v_heads), device=dev)
    _t(qkv_out, "qkv_out", d.dtype, (t, d.conv_dim))
    _t(g_out, "g_out", torch.float32, (t, d.n_v_heads))
    _t(beta_out, "beta_out", torch.float32, (t, d.n_v_heads))
    dd, pp = d.c(), params.c(d)
    st = lib.gdn_conv(ctypes.byref(dd), ctypes.byref(pp), n, _p(cu_d),
                      ctypes.c_void_p(cu_h.data_ptr()), _p(x), _p(a), _p(b), _p(conv_state_in),
                      _p(conv_state_out), _p(qkv_out), _p(g_out), _p(beta_out), _stream(dev))
    _check("gdn_conv", st)
    return qkv_out, g_out, beta_out


def prefill_workspace_size(d: Dims, cu_seqlens) -> int:
    lib = load()
    host = torch.tensor(list(cu_seqlens), dtype=torch.int32) if not isinstance(
        cu_seqlens, torch.Tensor) else cu_seqlens.detach().to("cpu", torch.int32).contiguous()
    out = ctypes.c_size_t(0)
    dd = d.c()
    _check("gdn_prefill_workspace_size",
           lib.gdn_prefill_workspace_size(ctypes.byref(dd), host.numel() - 1,
                                          ctypes.c_void_p(host.data_ptr()), ctypes.byref(out)))
    return int(out.value)


def prefill(d: Dims, params: Params, cu_seqlens, x, z, a, b, *, initial_state=None,
            final_state=None, conv_state_in=None, conv_state_out=None, out=None,
            workspace=None):
    """gdn_prefill over packed sequences.  Returns out [T, Hv*dv]."""
    lib = load()
    dev = x.device
    cu_d, cu_h = _cu_pair(cu_seqlens, dev)
    n = cu_h.numel() - 1
    t = int(cu_h[-1]) if n > 0 else 0
    vd = d.n_v_heads * d.d_v
    _t(x, "x", d.dtype, (t, d.conv_dim))
    _t(z, "z", d.dtype, (t, vd))
    _t(a, "a", d.dtype, (t, d.gate_width))
    _t(b, "b", d.dtype, (t, d.n_v_heads))
    st_shape = (n, d.n_v_heads, d.d_k, d.d_v)
    _t(initial_state, "initial_state", torch.float32, st_shape)
    _t(final_state, "final_state", torch.float32, st_shape)
    cs_shape = (n, d.conv_dim, d.conv_k - 1)
    _t(conv_state_in, "conv_state_in", d.dtype, cs_shape)
    _t(conv_state_out, "conv_state_out", d.dtype, cs_shape)
    out = out if out is not None else torch.empty((t, vd), dtype=d.dtype, device=dev)
    _t(out, "out", d.dtype, (t, vd))
    need = prefill_workspace_size(d, cu_h)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dd, pp = d.c(), params.c(d)
    st = lib.gdn_prefill(ctypes.byref(dd), ctypes.byref(pp), n, _p(cu_d),
                         ctypes.c_void_p(cu_h.data_ptr()), _p(x), _p(z), _p(a), _p(b),
                         _p(conv_state_in), _p(conv_state_out), _p(initial_state), _p(final_state),
                         _p(out), _p(workspace), ws_bytes, _stream(dev))
    _check("gdn_prefill", st)
    return out


class Proj:
    """Projection weights around the core, bf16 [out_features, in_features]."""

    def __init__(self, w_qkv, w_z, w_a, w_b, w_out):
        self.w_qkv, self.w_z, self.w_a, self.w_b, self.w_out = w_qkv, w_z, w_a, w_b, w_out
        self.hidden = int(w_qkv.shape[1])

    def c(self, d: "Dims") -> _Proj:
        vd = d.n_v_heads * d.d_v
        _t(self.w_qkv, "w_qkv", torch.bfloat16, (d.conv_dim, self.hidden))
        _t(self.w_z, "w_z", torch.bfloat16, (vd, self.hidden))
        _t(self.w_a, "w_a", torch.bfloat16, (d.n_v_heads, self.hidden))
        _t(self.w_b, "w_b", torch.bfloat16, (d.n_v_heads, self.hidden))
        _t(self.w_out, "w_out", torch.bfloat16, (self.hidden, vd))
        return _Proj(*(ctypes.c_void_p(w.data_ptr()) for w in
                       (self.w_qkv, self.w_z, self.w_a, self.w_b, self.w_out)))


def layer_prefill_workspace_size(d: Dims, hidden: int, cu_seqlens) -> int:
    lib = load()
    host = torch.tensor(list(cu_seqlens), dtype=torch.int32) if not isinstance(
        cu_seqlens, torch.Tensor) else cu_seqlens.detach().to("cpu", torch.int32).contiguous()
    out = ctypes.c_size_t(0)
    dd = d.c()
    _check("gdn_layer_prefill_workspace_size",
           lib.gdn_layer_prefill_workspace_size(ctypes.byref(dd), hidden, host.numel() - 1,
                                                ctypes.c_void_p(host.data_ptr()), ctypes.byref(out)))
    return int(out.value)


def layer_prefill(d: Dims, params: Params, proj: Proj, cu_seqlens, h, *, initial_state=None,
                  final_state=None, conv_state_in=None, conv_state_out=None, out=None,
                  workspace=None):
    """gdn_layer_prefill: h [T, hidden] bf16 -> returns h_out [T, hidden] bf16."""
    lib = load()
    dev = h.device
    cu_d, cu_h = _cu_pair(cu_seqlens, dev)
    n = cu_h.numel() - 1
    t = int(cu_h[-1]) if n > 0 else 0
    hid = proj.hidden
    _t(h, "h", torch.bfloat16, (t, hid))
    st_shape = (n, d.n_v_heads, d.d_k, d.d_v)
    _t(initial_state, "initial_state", torch.float32, st_shape)
    _t(final_state, "final_state", torch.float32, st_shape)
    cs_shape = (n, d.conv_dim, d.conv_k - 1)
    _t(conv_state_in, "conv_state_in", d.dtype, cs_shape)
    _t(conv_state_out, "conv_state_out", d.dtype, cs_shape)
    out = out if out is not None else torch.empty((t, hid), dtype=torch.bfloat16, device=dev)
    _t(out, "out", torch.bfloat16, (t, hid))
    need = layer_prefill_workspace_size(d, hid, cu_h)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    dd, pp, pj = d.c(), params.c(d), proj.c(d)
    st = lib.gdn_layer_prefill(ctypes.byref(dd), ctypes.byref(pp), ctypes.byref(pj), hid, n,
                               _p(cu_d), ctypes.c_void_p(cu_h.data_ptr()), _p(h),
                               _p(initial_state), _p(final_state), _p(conv_state_in),
                               _p(conv_state_out), _p(out), _p(workspace), ws_bytes, _stream(dev))
    _check("gdn_layer_prefill", st)
    return out


def decode(d: Dims, params: Params, x, z, a, b, state, conv_state=None, inter_states=None,
           out=None):
    """gdn_decode: x [N, T, CD] (or [N*T, CD] with T=1), state [N,Hv,dk,dv] fp32.

    Returns out [N, T, Hv*dv].  With ``inter_states`` [N,T,Hv,dk,dv] the state and
    conv state are read only; otherwise they are updated in place."""
    lib = load()
    dev = x.device
    if x.dim() == 2:
        x = x.unsqueeze(1)
    n, tt = x.shape[0], x.shape[1]
    vd = d.n_v_heads * d.d_v
    _t(x, "x", d.dtype, (n, tt, d.conv_dim))
    z = z.reshape(n, tt, vd) if z.dim() == 2 else z
    a = a.reshape(n, tt, d.gate_width) if a.dim() == 2 else a
    b = b.reshape(n, tt, d.n_v_heads) if b.dim() == 2 else b
    _t(z, "z", d.dtype, (n, tt, vd))
    _t(a, "a", d.dtype, (n, tt, d.gate_width))
    _t(b, "b", d.dtype, (n, tt, d.n_v_heads))
    _t(state, "state", torch.float32, (n, d.n_v_heads, d.d_k, d.d_v))
    _t(conv_state, "conv_state", d.dtype, (n, d.conv_dim, d.conv_k - 1))
    _t(inter_states, "inter_states", torch.float32, (n, tt, d.n_v_heads, d.d_k, d.d_v))
    out = out if out is not None else torch.empty((n, tt, vd), dtype=d.dtype, device=dev)
    _t(out, "out", d.dtype, (n, tt, vd))
    dd, pp = d.c(), params.c(d)
    st = lib.gdn_decode(ctypes.byref(dd), ctypes.byref(pp), n, tt, _p(x), _p(z), _p(a), _p(b),
                        _p(state), _p(conv_state), _p(inter_states), _p(out), _stream(dev))
    _check("gdn_decode", st)
    return out


def verify(d: Dims, params: Params, x, z, a, b, state, conv_state=None, out=None):
    """gdn_verify: x [N, T, CD]; state and conv_state are only read.

    Returns out [N, T, Hv*dv].  Replay the accepted prefix with ``prefill``."""
    lib = load()
    dev = x.device
    n, tt = x.shape[0], x.shape[1]
    vd = d.n_v_heads * d.d_v
    _t(x, "x", d.dtype, (n, tt, d.conv_dim))
    _t(z, "z", d.dtype, (n, tt, vd))
    _t(a, "a", d.dtype, (n, tt, d.gate_width))
    _t(b, "b", d.dtype, (n, tt, d.n_v_heads))
    _t(state, "state", torch.float32, (n, d.n_v_heads, d.d_k, d.d_v))
    _t(conv_state, "conv_state", d.dtype, (n, d.conv_dim, d.conv_k - 1))
    out = out if out is not None else torch.empty((n, tt, vd), dtype=d.dtype, device=dev)
    _t(out, "out", d.dtype, (n, tt, vd))
    dd, pp = d.c(), params.c(d)
    st = lib.gdn_verify(ctypes.byref(dd), ctypes.byref(pp), n, tt, _p(x), _p(z), _p(a), _p(b),
                        _p(state), _p(conv_state), _p(out), _stream(dev))
    _check("gdn_verify", st)
    return out


def decode_commit(d: Dims, accepted, x, inter_states, state, conv_state=None):
    """gdn_decode_commit: keep the first accepted[i] tokens of a verify call."""
    lib = load()
    dev = state.device
    n, tt = inter_states.shape[0], inter_states.shape[1]
    _t(accepted, "accepted", torch.int32, (n,))
    _t(x, "x", d.dtype, (n, tt, d.conv_dim))
    _t(inter_states, "inter_states", torch.float32, (n, tt, d.n_v_heads, d.d_k, d.d_v))
    _t(state, "state", torch.float32, (n, d.n_v_heads, d.d_k, d.d_v))
    _t(conv_state, "conv_state", d.dtype, (n, d.conv_dim, d.conv_k - 1))
    dd = d.c()
    st = lib.gdn_decode_commit(ctypes.byref(dd), n, tt, _p(accepted), _p(x), _p(inter_states),
                               _p(state), _p(conv_state), _stream(dev))
    _check("gdn_decode_commit", st)


__all__ = ["Dims", "Params", "GDNError", "load", "version", "timing_enable", "timing_report",
           "device_error", "sync_status",
           "conv", "prefill",
           "prefill_workspace_size", "decode", "verify", "decode_commit", "Proj",
           "layer_prefill_workspace_size", "layer_prefill", "EXPORTS", "LIB_PATH"]
