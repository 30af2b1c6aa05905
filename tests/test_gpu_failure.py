"""Failure detection on the GPU, made without faulting the GPU.

Two failure paths of a serving caller (cortiq-engine 0.8.76 pipeline.rs fails
closed: graph_failed -> clear_sequence_state; its test-only nll_test_fail_at
makes a step fail on purpose):

* a call fails on the host (GDN_FAULT lists its site): it returns
  GDN_ERR_INJECTED and leaves every device buffer as it was;
* a bounded device wait runs out: GDN_FAULT=stall_scan makes the fused
  tensor-core prefill's scan wait, for at most 1 ms, on a chunk flag that
  nothing sets.  The scan gives up, unwinds (it has issued no copy or MMA
  at that point and releases its tensor memory), and records wait code 11;
  gdn_sync_status then reports GDN_ERR_TIMEOUT, and the next call on the same
  context computes correct results again.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_mixer_gb300 as gdn
from gated_deltanet_linear_mixer_gb300 import workloads
from gdn_cases import TOL, dims, gpu_prefill, rel_err, run_oracle, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_mixer_gb300 import _build
    _build.build()
    gdn.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gdn.device_error(reset=True)
    yield
    gdn.device_error(reset=True)


def _case():
    # a small batch: its scan clusters leave room for prep, so it takes the fused launch
    return workloads.generate("fail", n_k_heads=2, n_v_heads=2, d_k=128, d_v=128, conv_k=4,
                              dtype="bf16", act="silu", seed=51, lengths=[150, 64, 65],
                              state_std=0.05, conv_state_std=1.0)


@pytest.mark.parametrize("site", ["prefill", "all"])
def test_injected_prefill_leaves_device_buffers_untouched(monkeypatch, site):
    case = _case()
    d, _ = dims(case)
    t = upload(case)
    n = case.n_seq
    st_in = t["state"].clone()
    st_out = torch.full((n, d.n_v_heads, d.d_k, d.d_v), 7.0, device="cuda")
    cs_out = torch.full((n, d.conv_dim, d.conv_k - 1), 7.0, dtype=d.dtype, device="cuda")
    out = torch.full((case.n_tokens, d.n_v_heads * d.d_v), 7.0, dtype=d.dtype, device="cuda")
    monkeypatch.setenv("GDN_FAULT", site)
    with pytest.raises(gdn.GDNError) as e:
        gdn.prefill(d, t["params"], case.cu_seqlens, t["x"], t["z"], t["a"], t["b"],
                    initial_state=st_in, final_state=st_out, conv_state_in=t["conv_state"],
                    conv_state_out=cs_out, out=out)
    assert e.value.status == gdn.GDN_ERR_INJECTED
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(st_out == 7.0) and torch.all(cs_out == 7.0)
    assert torch.equal(st_in, t["state"])
    monkeypatch.delenv("GDN_FAULT")
    gdn.sync_status()  # nothing ran, nothing failed


def test_bounded_scan_wait_runs_out_and_is_reported(monkeypatch):
    case = _case()
    monkeypatch.setenv("GDN_FAULT", "stall_scan")
    gpu_prefill(case)  # enqueued fine; the scan gives up on the device
    with pytest.raises(gdn.GDNError) as e:
        gdn.sync_status()
    assert e.value.status == gdn.GDN_ERR_TIMEOUT
    assert "wait code 11" in str(e.value)
    gdn.sync_status()  # the word was cleared by the report
    # the context is still usable: the same call without the hook is correct
    monkeypatch.delenv("GDN_FAULT")
    got = gpu_prefill(case)
    gdn.sync_status()
    ref = run_oracle(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_stall_hook_does_not_touch_the_token_recurrent_path(monkeypatch):
    """The hook only acts on the fused tensor-core launch: an fp32 prefill (the
    token-recurrent kernel, no cross-CTA waits) runs normally with it set."""
    case = workloads.config(0)
    monkeypatch.setenv("GDN_FAULT", "stall_scan")
    got = gpu_prefill(case)
    gdn.sync_status()
    ref = run_oracle(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["f32"]
    assert np.isfinite(got["state"].cpu().numpy()).all()
