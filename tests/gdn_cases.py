"""Shared test helpers: upload a synthetic case, run the CUDA path through the
C ABI, run the oracle on the same values, and measure the error.

Error metric (the tolerance statement of the workloads): max |gpu - ref| divided
by the RMS of the reference tensor, per tensor.  Tolerances: 1e-4 for fp32
activations, 2e-2 for bf16 activations with fp32 state.

A result stored as bf16 carries the rounding of its own storage: half a bf16
ulp, up to 2^-9 of the value, which for the heavy-tailed gated outputs (values
up to ~50x the RMS) is several 1e-2 of the RMS by itself.  For bf16-stored
tensors the error counted is therefore what exceeds that half ulp of the stored
value: max(0, |gpu - ref| - ulp_bf16(gpu)/2).  fp32 tensors are compared as is.
"""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_mixer_gb300 as gdn
import oracle

TOL = {"f32": 1e-4, "bf16": 2e-2}


def bf16_half_ulp(v):
    """Half the bf16 ulp of each (bf16-representable) value; 0 for zeros."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, np.exp2(e - 8.0), 0.0)


def rel_err(got, ref) -> float:
    is_bf16 = isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16
    got = got.detach().float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref ** 2)))
    if not np.all(np.isfinite(got)):
        return float("inf")
    diff = np.abs(got - ref)
    if is_bf16:
        diff = np.maximum(diff - bf16_half_ulp(got), 0.0)
    return float(np.max(diff) / max(rms, 1e-30))


def dims(case):
    """Library and oracle geometry of a case; a case may carry head_map and
    decay_form (the ABI options), else the defaults."""
    tdt = torch.bfloat16 if case.dtype == "bf16" else torch.float32
    opt = dict(head_map=getattr(case, "head_map", "contiguous"),
               decay_form=getattr(case, "decay_form", "A_log"),
               per_channel_decay=getattr(case, "per_channel_decay", False))
    d = gdn.Dims(case.n_k_heads, case.n_v_heads, case.d_k, case.d_v, case.conv_k, tdt, case.act,
                 **opt)
    od = oracle.Dims(case.n_k_heads, case.n_v_heads, case.d_k, case.d_v, case.conv_k, case.act,
                     **opt)
    return d, od


def upload(case, device="cuda"):
    tdt = torch.bfloat16 if case.dtype == "bf16" else torch.float32

    def act(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=tdt).contiguous()

    def f32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=torch.float32).contiguous()

    t = dict(x=act(case.x), z=act(case.z), a=act(case.a), b=act(case.b),
             conv_state=act(case.conv_state), state=f32(case.state),
             cu=torch.from_numpy(case.cu_seqlens).to(device))
    t["params"] = gdn.Params(f32(case.conv_w), f32(case.A_log), f32(case.dt_bias), f32(case.norm_w))
    return t


def run_oracle(case, want_inter=False, want_stages=False):
    _, od = dims(case)
    return oracle.gdn(od, case.cu_seqlens, case.x, case.z, case.a, case.b, case.conv_w,
                      case.A_log, case.dt_bias, case.norm_w, case.conv_state, case.state,
                      want_inter=want_inter, want_stages=want_stages)


def gpu_prefill(case, t=None, in_place=False, workspace=None):
    d, _ = dims(case)
    t = t or upload(case)
    n = case.n_seq
    dev = t["x"].device
    if in_place:
        st_in = t["state"] if t["state"] is not None else torch.zeros(
            (n, d.n_v_heads, d.d_k, d.d_v), device=dev)
        st_out = st_in
        cs_in = t["conv_state"] if t["conv_state"] is not None else torch.zeros(
            (n, d.conv_dim, d.conv_k - 1), dtype=d.dtype, device=dev)
        cs_out = cs_in
    else:
        st_in = t["state"]
        st_out = torch.full((n, d.n_v_heads, d.d_k, d.d_v), float("nan"), device=dev)
        cs_in = t["conv_state"]
        cs_out = torch.full((n, d.conv_dim, d.conv_k - 1), float("nan"), dtype=d.dtype, device=dev)
    out = torch.full((case.n_tokens, d.n_v_heads * d.d_v), float("nan"), dtype=d.dtype, device=dev)
    gdn.prefill(d, t["params"], case.cu_seqlens, t["x"], t["z"], t["a"], t["b"],
                initial_state=st_in, final_state=st_out, conv_state_in=cs_in,
                conv_state_out=cs_out, out=out, workspace=workspace)
    torch.cuda.synchronize()
    return {"out": out, "state": st_out, "conv_state": cs_out}


def gpu_decode(case, t=None, inter=False):
    d, _ = dims(case)
    t = t or upload(case)
    n, tt = case.n_seq, case.tokens_per_seq
    dev = t["x"].device
    state = t["state"].clone()
    cs = None if t["conv_state"] is None else t["conv_state"].clone()
    inter_t = None
    if inter:
        inter_t = torch.full((n, tt, d.n_v_heads, d.d_k, d.d_v), float("nan"), device=dev)
    out = torch.full((n, tt, d.n_v_heads * d.d_v), float("nan"), dtype=d.dtype, device=dev)
    gdn.decode(d, t["params"], t["x"].view(n, tt, -1), t["z"].view(n, tt, -1),
               t["a"].view(n, tt, -1), t["b"].view(n, tt, -1), state, cs, inter_t, out)
    torch.cuda.synchronize()
    return {"out": out.view(n * tt, -1), "state": state, "conv_state": cs, "inter": inter_t}
