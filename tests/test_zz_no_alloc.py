"""The prefill entry point that allocates nothing (gdn_prefill_noalloc).

Callers such as an engine plugin handed only its inputs and outputs, or a
serving loop whose device memory is fixed before it starts, cannot allocate
the workspace gdn_prefill asks for; gdn_prefill_noalloc runs the same prefill
on a built-in device array instead.  These tests call it through the C ABI
directly and check it against gdn_prefill on the same inputs and against the
oracle, on two calls in a row (the second call finds the first call's contents
in the shared array).

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mixer_gb300 as gdn
from gated_deltanet_linear_mixer_gb300 import workloads
from gdn_cases import TOL, dims, rel_err, run_oracle, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_mixer_gb300 import _build
    _build.build()
    gdn.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _case(seed, lengths):
    return workloads.generate("noalloc", n_k_heads=16, n_v_heads=32, d_k=128, d_v=128, conv_k=4,
                              dtype="bf16", act="silu", seed=seed, lengths=lengths,
                              state_std=0.05, conv_state_std=1.0)


def _noalloc(case, t):
    """One gdn_prefill_noalloc call through ctypes; returns (status, out, state, conv)."""
    lib = gdn.load()
    d, _ = dims(case)
    n, dev = case.n_seq, t["x"].device
    cu_h = torch.from_numpy(case.cu_seqlens.astype(np.int32).copy())
    st_out = torch.full((n, d.n_v_heads, d.d_k, d.d_v), float("nan"), device=dev)
    cs_out = torch.full((n, d.conv_dim, d.conv_k - 1), float("nan"), dtype=d.dtype, device=dev)
    out = torch.full((case.n_tokens, d.n_v_heads * d.d_v), float("nan"), dtype=d.dtype, device=dev)
    dd, pp = d.c(), t["params"].c(d)
    p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    status = lib.gdn_prefill_noalloc(
        ctypes.byref(dd), ctypes.byref(pp), n, p(t["cu"]), ctypes.c_void_p(cu_h.data_ptr()),
        p(t["x"]), p(t["z"]), p(t["a"]), p(t["b"]), p(t["conv_state"]), p(cs_out),
        p(t["state"]), p(st_out), p(out),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return status, out, st_out, cs_out


def _regular(case, t):
    d, _ = dims(case)
    n, dev = case.n_seq, t["x"].device
    st_out = torch.empty((n, d.n_v_heads, d.d_k, d.d_v), device=dev)
    cs_out = torch.empty((n, d.conv_dim, d.conv_k - 1), dtype=d.dtype, device=dev)
    out = gdn.prefill(d, t["params"], case.cu_seqlens, t["x"], t["z"], t["a"], t["b"],
                      initial_state=t["state"], final_state=st_out,
                      conv_state_in=t["conv_state"], conv_state_out=cs_out)
    torch.cuda.synchronize()
    return out, st_out, cs_out


def test_noalloc_prefill_matches_the_workspace_entry_point_on_two_calls():
    """Two calls in a row with different inputs and sequence layouts; each must
    match gdn_prefill (same kernels, caller-owned workspace) and the oracle within
    the suite's bf16 tolerance, and the conv history exactly."""
    gdn.device_error(reset=True)
    for seed, lengths in ((41, [200, 64, 131]), (42, [77, 1, 256])):
        case = _case(seed, lengths)
        t = upload(case)
        status, out, st, cs = _noalloc(case, t)
        assert status == gdn.GDN_OK, gdn.load().gdn_last_error().decode()
        ref_out, ref_st, ref_cs = _regular(case, t)
        assert rel_err(out, ref_out.float().cpu().numpy()) < TOL["bf16"]
        assert rel_err(st, ref_st.cpu().numpy()) < TOL["bf16"]
        assert torch.equal(cs, ref_cs)
        oracle_ref = run_oracle(case)
        assert rel_err(out, oracle_ref["out"]) <= TOL["bf16"]
        assert rel_err(st, oracle_ref["state"]) <= TOL["bf16"]
        assert rel_err(cs.float(), oracle_ref["conv_state"]) == 0.0
    assert gdn.device_error(reset=True) == 0


def test_noalloc_call_allocates_no_device_memory():
    """After a first call (set-up: it makes the built-in array resident and looks
    up its address), a call with another sequence layout changes neither the
    device's free memory nor PyTorch's allocations: the call itself allocates
    nothing.  Every buffer it is handed is allocated before the measurement."""
    case_a, case_b = _case(44, [90, 30]), _case(45, [129, 3, 64])
    ta, tb = upload(case_a), upload(case_b)
    status, _, _, _ = _noalloc(case_a, ta)  # set-up call
    assert status == gdn.GDN_OK, gdn.load().gdn_last_error().decode()
    lib = gdn.load()
    d, _ = dims(case_b)
    n, dev = case_b.n_seq, tb["x"].device
    cu_h = torch.from_numpy(case_b.cu_seqlens.astype(np.int32).copy())
    st_out = torch.empty((n, d.n_v_heads, d.d_k, d.d_v), device=dev)
    cs_out = torch.empty((n, d.conv_dim, d.conv_k - 1), dtype=d.dtype, device=dev)
    out = torch.empty((case_b.n_tokens, d.n_v_heads * d.d_v), dtype=d.dtype, device=dev)
    dd, pp = d.c(), tb["params"].c(d)
    p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(2):
        status = lib.gdn_prefill_noalloc(
            ctypes.byref(dd), ctypes.byref(pp), n, p(tb["cu"]), ctypes.c_void_p(cu_h.data_ptr()),
            p(tb["x"]), p(tb["z"]), p(tb["a"]), p(tb["b"]), p(tb["conv_state"]), p(cs_out),
            p(tb["state"]), p(st_out), p(out), stream)
        assert status == gdn.GDN_OK, lib.gdn_last_error().decode()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0
    ref_out, ref_st, _ = _regular(case_b, tb)
    assert rel_err(out, ref_out.float().cpu().numpy()) < TOL["bf16"]
    assert rel_err(st_out, ref_st.cpu().numpy()) < TOL["bf16"]


def test_noalloc_per_channel_decay_matches_the_oracle():
    """Per-channel decay through the entry point that allocates nothing: its
    chunked form (its own prep, wider workspace rows) on the built-in array."""
    case = workloads.with_per_channel_decay(_case(46, [150, 33]), seed=47)
    t = upload(case)
    status, out, st, cs = _noalloc(case, t)
    assert status == gdn.GDN_OK, gdn.load().gdn_last_error().decode()
    ref = run_oracle(case)
    assert rel_err(out, ref["out"]) <= TOL["bf16"]
    assert rel_err(st, ref["state"]) <= TOL["bf16"]
    assert rel_err(cs.float(), ref["conv_state"]) == 0.0
    assert gdn.device_error(reset=True) == 0


def test_noalloc_refuses_a_layout_beyond_its_scratch():
    lib = gdn.load()
    limit = int(lib.gdn_prefill_noalloc_scratch_bytes())
    case = _case(43, [64])
    d, _ = dims(case)
    t_big = 4096
    cu_h = torch.tensor([0, t_big], dtype=torch.int32)
    assert gdn.prefill_workspace_size(d, cu_h) > limit
    t = upload(case)
    dd, pp = d.c(), t["params"].c(d)
    dummy = ctypes.c_void_p(t["x"].data_ptr())  # never dereferenced: the call is refused first
    status = lib.gdn_prefill_noalloc(
        ctypes.byref(dd), ctypes.byref(pp), 1, ctypes.c_void_p(t["cu"].data_ptr()),
        ctypes.c_void_p(cu_h.data_ptr()), dummy, dummy, dummy, dummy, None, None, None, None,
        dummy, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 4  # GDN_ERR_WORKSPACE
    assert b"scratch" in lib.gdn_last_error()
