"""bench.py's host logic, with no GPU: the algorithmic bytes and useful flops
that the roofline figures divide by, checked against counts made by hand from
the workload shapes, and the JSON line of the reference arm."""
import json
import os
import subprocess
import sys

import pytest

import bench
from gated_deltanet_linear_mixer_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# The Qwen3-Next-shaped head geometry of every bench workload.
HV, DK, DV, CD, KEEP = 32, 128, 128, 8192, 3
STATE = 4 * HV * DK * DV                      # fp32 state of one sequence
CONV = 2 * CD * KEEP                          # bf16 conv history of one sequence
ACT = 2 * (CD + HV * DV + 2 * HV + HV * DV)   # x, z, a, b in and out, per token


def _runner(key):
    """A Runner with its workload but no device buffers (host logic only)."""
    r = bench.Runner.__new__(bench.Runner)
    r.key, r.case = key, workloads.config(bench.WORKLOADS[key])
    return r


def test_hand_counts():
    assert (STATE, CONV, ACT) == (2_097_152, 49_152, 32_896)


def test_prefill_bytes():
    r = _runner("prefill")  # zero initial state: final state and history out
    assert r.algorithmic_bytes() == 4096 * ACT + STATE + CONV


def test_decode_bytes_per_sequence_step():
    r = _runner("decode")  # state and history read and written once each
    per_seq = ACT + 2 * STATE + 2 * CONV
    assert per_seq == 4_325_504
    assert r.algorithmic_bytes() == 256 * per_seq


def test_spec_verify_bytes_per_sequence():
    r = _runner("spec_verify")  # state read once, four intermediates written, history read
    per_seq = 4 * ACT + 5 * STATE + CONV
    assert per_seq == 10_666_496
    assert r.algorithmic_bytes() == 64 * per_seq


def test_spec_replay_launch_bytes():
    r = _runner("spec_replay")
    # verify: 4 drafts in, state and history read; replay of 2 accepted tokens:
    # their inputs again, state and history read and written
    step = 64 * (4 * ACT + 2 * ACT + 3 * STATE + 3 * CONV)
    assert r.algorithmic_bytes() == step
    # the recurrent kernel runs twice a step; the history kernel takes its rows
    assert r.kernel_bytes("conv_state") == 2 * 64 * CONV
    assert r.kernel_bytes("recurrent", ("recurrent", "conv_state")) == (step - 2 * 64 * CONV) / 2


def test_varlen_bytes():
    r = _runner("varlen")  # initial state in, final state out, history out
    c = r.case
    assert r.algorithmic_bytes() == c.n_tokens * ACT + c.n_seq * (2 * STATE + CONV)


def test_prefill_useful_flops():
    r = _runner("prefill")
    per_token_head = 6 * DK * DV + 64 * (3 * DK + 2 * DV) + 64 * 64 / 3
    assert round(per_token_head) == 140_629
    assert r.useful_flops() == pytest.approx(per_token_head * HV * 4096)
    assert r.useful_flops() == pytest.approx(18.4326e9, rel=1e-4)


def test_reference_arm_line():
    """`bench.py --impl reference` prints one JSON line with the contract's keys;
    it runs the oracle on host cores only."""
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def _kda_runner():
    r = bench.Runner.__new__(bench.Runner)
    r.key = "kda_prefill"
    r.case = workloads.with_per_channel_decay(workloads.config(bench.WORKLOADS["kda_prefill"]), bench.KDA_SEED)
    return r


def test_kda_prefill_bytes():
    """Per-channel decay: the gate input a is [T, Hv*dk] instead of [T, Hv]."""
    r = _kda_runner()
    act = ACT + 2 * HV * (DK - 1)
    assert act == 41_024
    assert r.algorithmic_bytes() == 4096 * act + STATE + CONV


def test_kda_kernel_flops_split_the_chunked_form():
    """The prep's and the scan's shares of the contractions add up to the
    chunked form's useful flops."""
    r = _kda_runner()
    prep, scan = r.kernel_flops("chunk_prep_kda"), r.kernel_flops("chunk_scan_kda")
    assert prep == pytest.approx((64 * (3 * DK + DV) + 64 * 64 / 3) * HV * 4096)
    assert scan == pytest.approx((6 * DK * DV + 64 * DV) * HV * 4096)
    assert prep + scan == pytest.approx(r.useful_flops())
