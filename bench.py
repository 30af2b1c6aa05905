#!/usr/bin/env python3
"""Benchmark of the GDN mixer core on one GB300 (or N replicas under torchrun).

Prints ONE JSON line.  The headline is prefill tokens/s on the T=4096,
Hk=16, Hv=32, d_k=d_v=128 bf16 workload ("value"); the same line carries
decode tokens/s (256 sequences x 1 token), the packed variable-length prefill
(16 sequences, lengths U{128..8192}) and the speculative-verify decode
(64 sequences x 4 tokens, every intermediate state emitted), each with its
roofline against the measured peaks, the dominant kernel's per-launch time from
CUDA events recorded by libgdn on the launching stream, and an end-to-end
figure through the public API with pinned host buffers.

``--impl reference`` times the CPU oracle instead (the only baseline: the pages
publish no GPU implementation of this core): the float build of its C source,
one whole prefill workload per step.  The same build, on the same workloads, is
each GPU line's ``cpu_baseline``.

Timing: W untimed warm-up steps, then K timed steps between a barrier and a
device synchronize; a 256 MiB buffer (2x L2) is written between timed steps
and each step is bracketed by CUDA events on the launching stream.  The
per-kernel durations come from a second pass of the same K steps with
libgdn's per-launch events switched on, which the step time leaves out.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s and decode tokens/s (1 GB300) + % of roofline"
# DRAM bytes (read + write) per launch of a workload's dominant kernel, from an
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of the kernel as it
# is now: (bytes, where they come from).  A capture of a smaller case is scaled
# by the units it processes, and the source says so.  An entry is removed when
# its kernel changes, until it is captured again.
TRAFFIC = {
    ("prefill", "chunk_fused"): (259_900_000 + 202_250_000, "ncu capture of this workload's launch"),
    ("layer", "chunk_fused"): (259_900_000 + 202_250_000,
                               "ncu capture of the same launch in the T=4096 prefill workload"),
    # 64-sequence decode step; the traffic is per sequence: x 256/64
    ("decode", "recurrent"): ((139_130_000 + 72_380_000) * 4,
                              "ncu capture of the 64-sequence decode step, scaled x 256/64"),
    ("spec_verify", "recurrent"): (144_420_000 + 476_470_000, "ncu capture of this workload's launch"),
    # the step's two launches under one name: the read-only verify and the replay
    ("spec_replay", "recurrent"): (((143_920_000 + 3_660_000) + (140_710_000 + 73_090_000)) // 2,
                                   "ncu captures of the step's two launches (verify, replay), averaged"),
    ("kda_prefill", "chunk_prep_kda"): (168_550_000 + 244_610_000, "ncu capture of this workload's launch"),
    # 16 sequences of 128..1024 tokens (149 chunks); the traffic is per chunk: x 1015/149
    ("varlen", "chunk_scan"): (round((657_530_000 + 91_200_000) * 1015 / 149),
                               "ncu capture of a 149-chunk varlen case, scaled x 1015/149 chunks"),
}
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ----------------------------------------------------------------- workloads
# Algorithmic bytes: what the core must read and write at minimum (inputs once,
# outputs once, states once each way).  Activations are bf16.

def _act_bytes_per_token(c):
    cd, vd, hv = c.conv_dim, c.n_v_heads * c.d_v, c.n_v_heads
    gates = hv * (c.d_k if getattr(c, "per_channel_decay", False) else 1)  # a: per value head or channel
    return 2 * (cd + vd + gates + hv + vd)  # x, z, a, b in; out


def _state_bytes(c):
    return 4 * c.n_v_heads * c.d_k * c.d_v


def _conv_state_bytes(c):
    return 2 * c.conv_dim * (c.conv_k - 1)


WORKLOADS = {
    # key: (config index, description)
    "prefill": 1,
    "decode": 2,
    "varlen": 3,
    "spec_verify": 4,
    "spec_replay": 4,   # the same drafts, verified read-only, accepted prefix replayed
    "layer": 1,         # the T=4096 prefill inside a whole layer: in_proj -> core -> out_proj
    "kda_prefill": 1,   # the T=4096 prefill with one decay per key channel
}
KDA_SEED = 98           # gate draw of kda_prefill (a [T, Hv*dk], dt_bias [Hv*dk])
LAYER_HIDDEN = 2048     # model width of the layer workload (Qwen3-Next's hidden size)
REPLAY_ACCEPTED = 2     # tokens of every sequence's 4 drafts accepted in spec_replay


class Runner:
    """Holds device buffers of one workload and runs one step of it."""

    def __init__(self, key, case, device):
        import torch
        import gated_deltanet_linear_mixer_gb300 as gdn
        self.key, self.case, self.dev = key, case, device
        self.gdn, self.torch = gdn, torch
        c = case
        self.d = gdn.Dims(c.n_k_heads, c.n_v_heads, c.d_k, c.d_v, c.conv_k, torch.bfloat16, c.act,
                          per_channel_decay=getattr(c, "per_channel_decay", False))
        bf = lambda a: torch.from_numpy(a).to(device=device, dtype=torch.bfloat16)  # noqa: E731
        f32 = lambda a: torch.from_numpy(a).to(device=device, dtype=torch.float32)  # noqa: E731
        self.x, self.z, self.a, self.b = bf(c.x), bf(c.z), bf(c.a), bf(c.b)
        self.params = gdn.Params(f32(c.conv_w), f32(c.A_log), f32(c.dt_bias), f32(c.norm_w))
        n = c.n_seq
        self.cu_host = torch.from_numpy(c.cu_seqlens.copy())
        self.cu_dev = self.cu_host.to(device)
        vd = c.n_v_heads * c.d_v
        self.out = torch.empty((c.n_tokens, vd), dtype=torch.bfloat16, device=device)
        self.state0 = None if c.state is None else f32(c.state)
        self.state = None if c.state is None else self.state0.clone()
        self.conv0 = None if c.conv_state is None else bf(c.conv_state)
        self.conv = None if c.conv_state is None else self.conv0.clone()
        self.final = torch.empty((n, c.n_v_heads, c.d_k, c.d_v), device=device)
        self.conv_out = torch.empty((n, c.conv_dim, c.conv_k - 1), dtype=torch.bfloat16, device=device)
        self.inter = None
        if key == "spec_verify":
            self.inter = torch.empty((n, c.tokens_per_seq, c.n_v_heads, c.d_k, c.d_v), device=device)
        if key == "spec_replay":  # the accepted prefixes, packed, and their cu_seqlens
            t, j = c.tokens_per_seq, REPLAY_ACCEPTED
            take = lambda u: u.view(n, t, -1)[:, :j].reshape(n * j, -1).contiguous()  # noqa: E731
            self.rx, self.rz, self.ra, self.rb = (take(u) for u in (self.x, self.z, self.a, self.b))
            self.rcu_host = torch.arange(0, n * j + 1, j, dtype=torch.int32)
            self.rcu_dev = self.rcu_host.to(device)
            self.rout = torch.empty((n * j, vd), dtype=torch.bfloat16, device=device)
        if key == "layer":  # synthetic bf16 weights ~N(0, 1/in_features), hidden states ~N(0,1)
            rng = np.random.default_rng(5)
            shapes = {"w_qkv": (c.conv_dim, LAYER_HIDDEN), "w_z": (vd, LAYER_HIDDEN),
                      "w_a": (c.n_v_heads, LAYER_HIDDEN), "w_b": (c.n_v_heads, LAYER_HIDDEN),
                      "w_out": (LAYER_HIDDEN, vd)}
            w = {k: bf(rng.normal(0, 1 / np.sqrt(v[1]), size=v).astype(np.float32))
                 for k, v in shapes.items()}
            self.proj = gdn.Proj(w["w_qkv"], w["w_z"], w["w_a"], w["w_b"], w["w_out"])
            self.h = bf(rng.normal(size=(c.n_tokens, LAYER_HIDDEN)).astype(np.float32))
            self.layer_out = torch.empty_like(self.h)
            self.layer_ws = torch.empty(gdn.layer_prefill_workspace_size(self.d, LAYER_HIDDEN,
                                                                         self.cu_host),
                                        dtype=torch.uint8, device=device)
        ws = gdn.prefill_workspace_size(self.d, self.cu_host) if c.mode == "prefill" else 0
        self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=device)

    # -- one step through the public API (device-resident inputs)
    def step(self):
        gdn, c = self.gdn, self.case
        if self.key == "layer":
            gdn.layer_prefill(self.d, self.params, self.proj, (self.cu_dev, self.cu_host), self.h,
                              initial_state=self.state0, final_state=self.final,
                              conv_state_out=self.conv_out, out=self.layer_out,
                              workspace=self.layer_ws)
        elif self.key == "spec_replay":
            n, t = c.n_seq, c.tokens_per_seq
            gdn.verify(self.d, self.params, self.x.view(n, t, -1), self.z.view(n, t, -1),
                       self.a.view(n, t, -1), self.b.view(n, t, -1), self.state, self.conv,
                       self.out.view(n, t, -1))
            gdn.prefill(self.d, self.params, (self.rcu_dev, self.rcu_host), self.rx, self.rz,
                        self.ra, self.rb, initial_state=self.state, final_state=self.state,
                        conv_state_in=self.conv, conv_state_out=self.conv, out=self.rout,
                        workspace=self.ws)
        elif c.mode == "prefill":
            gdn.prefill(self.d, self.params, (self.cu_dev, self.cu_host), self.x, self.z, self.a,
                        self.b, initial_state=self.state0, final_state=self.final,
                        conv_state_in=None, conv_state_out=self.conv_out, out=self.out,
                        workspace=self.ws)
        else:
            n, t = c.n_seq, c.tokens_per_seq
            gdn.decode(self.d, self.params, self.x.view(n, t, -1), self.z.view(n, t, -1),
                       self.a.view(n, t, -1), self.b.view(n, t, -1), self.state, self.conv,
                       self.inter, self.out.view(n, t, -1))

    @property
    def tokens(self):
        return self.case.n_tokens

    def algorithmic_bytes(self):
        c = self.case
        act = _act_bytes_per_token(c) * c.n_tokens
        n = c.n_seq
        if self.key in ("prefill", "kda_prefill"):  # zero initial state (not read); final state +
            return act + n * (_state_bytes(c) + _conv_state_bytes(c))  # conv state out
        if self.key == "layer":        # h in, h_out, the weights once, final state + conv state out
            vd = c.n_v_heads * c.d_v
            w = 2 * LAYER_HIDDEN * (c.conv_dim + 2 * vd + 2 * c.n_v_heads)
            return 4 * LAYER_HIDDEN * c.n_tokens + w + n * (_state_bytes(c) + _conv_state_bytes(c))
        if self.key == "varlen":       # initial state in, final state out, conv state out
            return act + n * (2 * _state_bytes(c) + _conv_state_bytes(c))
        if self.key == "decode":       # state and conv state read and written in place
            return act + n * (2 * _state_bytes(c) + 2 * _conv_state_bytes(c))
        if self.key == "spec_verify":  # state read once, T states written, conv state read
            return act + n * ((1 + c.tokens_per_seq) * _state_bytes(c) + _conv_state_bytes(c))
        if self.key == "spec_replay":  # verify: state and history read; replay of the accepted
            # prefix: its inputs read once more, state and history read and written
            return (act + _act_bytes_per_token(c) * n * REPLAY_ACCEPTED
                    + n * (3 * _state_bytes(c) + 3 * _conv_state_bytes(c)))
        raise KeyError(self.key)

    def kernel_bytes(self, name, kernels=()):
        """Algorithmic bytes of one launch of kernel `name` (for the roofline).

        A separate conv-state kernel, when the step launches one, is charged the
        K-1 history rows; the step's other kernels share the rest."""
        c = self.case
        conv = c.n_seq * _conv_state_bytes(c)
        hist = {"prefill": conv, "varlen": conv, "decode": 2 * conv, "spec_verify": 0,
                "spec_replay": 2 * conv, "layer": conv, "kda_prefill": conv}[self.key]
        if name == "conv_state":
            return hist
        rest = self.algorithmic_bytes() - (hist if "conv_state" in kernels else 0)
        # spec_replay launches the recurrent kernel twice a step (verify, replay)
        return rest / 2 if self.key == "spec_replay" else rest

    def useful_flops(self, chunk=64, with_proj=True):
        """Useful flops of the chunked form per step (prefill), else of the recurrence;
        the layer workload adds its projections (in_proj: CD + Hv*dv + 2 Hv outputs,
        out_proj: hidden outputs from Hv*dv) unless with_proj is False."""
        c = self.case
        dk, dv = c.d_k, c.d_v
        if c.mode == "prefill":
            per_tok_head = 6 * dk * dv + chunk * (3 * dk + 2 * dv) + chunk * chunk / 3
        else:
            per_tok_head = 5 * dk * dv
        flops = per_tok_head * c.n_v_heads * c.n_tokens
        if self.key == "layer" and with_proj:
            vd = c.n_v_heads * dv
            flops += 2 * c.n_tokens * LAYER_HIDDEN * (c.conv_dim + 2 * vd + 2 * c.n_v_heads)
        return flops

    def kernel_flops(self, name, chunk=64):
        """Useful flops of one launch of a chunked-form kernel that does part of
        the contractions (the per-channel decay form's two launches): its prep
        forms the Gram matrices, the solve and [W | U~] = T [K | V] (per token
        and value head C (3 dk + dv) + C^2 / 3), its scan the state and output
        products (6 dk dv + C dv); the two add up to useful_flops()."""
        c = self.case
        dk, dv = c.d_k, c.d_v
        per = {"chunk_prep_kda": chunk * (3 * dk + dv) + chunk * chunk / 3,
               "chunk_scan_kda": 6 * dk * dv + chunk * dv}[name]
        return per * c.n_v_heads * c.n_tokens

    # -- end to end: pinned host buffers, H2D of the step's inputs, the call,
    # D2H of the step's outputs, pipelined as a serving loop runs them: the
    # inputs of step i+1 are copied in and the output of step i-1 is read back
    # on two copy streams while step i computes (two device buffer sets).
    def setup_e2e(self):
        torch = self.torch
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())  # noqa: E731
        self.in_names = ["h"] if self.key == "layer" else ["x", "z", "a", "b"]
        # the step's result read back by the caller: the mixer (or layer) output
        # (states stay resident on the device for the next call)
        self.out_names = ["layer_out"] if self.key == "layer" else ["out"]
        self.sets = []
        for k in range(2):
            d_in = {n: getattr(self, n) if k == 0 else getattr(self, n).clone() for n in self.in_names}
            d_out = {n: getattr(self, n) if k == 0 else torch.empty_like(getattr(self, n))
                     for n in self.out_names}
            h_in = {n: pin(t) for n, t in d_in.items()}
            h_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in d_out.items()}
            self.sets.append((d_in, d_out, h_in, h_out))
        self.h2d = sum(t.numel() * t.element_size() for t in self.sets[0][2].values())
        self.d2h = sum(t.numel() * t.element_size() for t in self.sets[0][3].values())
        self.s_in, self.s_out = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
        self.ev_in, self.ev_done, self.ev_read = ev(), ev(), ev()
        self.e2e_i = 0

    def e2e_step(self, stream):
        """One pipelined step on buffer set i % 2; `stream` is the compute stream."""
        torch, k = self.torch, self.e2e_i % 2
        d_in, d_out, h_in, h_out = self.sets[k]
        if self.e2e_i >= 2:
            self.s_in.wait_event(self.ev_done[k])   # step i-2 has read this input set
        with torch.cuda.stream(self.s_in):
            for n in self.in_names:
                d_in[n].copy_(h_in[n], non_blocking=True)
        self.ev_in[k].record(self.s_in)
        stream.wait_event(self.ev_in[k])
        if self.e2e_i >= 2:
            stream.wait_event(self.ev_read[k])      # step i-2's output has been read back
        for n in self.in_names + self.out_names:
            setattr(self, n, (d_in | d_out)[n])
        self.step()
        self.ev_done[k].record(stream)
        self.s_out.wait_event(self.ev_done[k])
        with torch.cuda.stream(self.s_out):
            for n in self.out_names:
                h_out[n].copy_(d_out[n], non_blocking=True)
        self.ev_read[k].record(self.s_out)
        self.e2e_i += 1


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index, self.samples, self.proc = index, [], None
        self._thr = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._thr = threading.Thread(target=self._read, daemon=True)
        self._thr.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        rows = [p for (ts, p) in self.samples if (t0 is None or ts >= t0) and (t1 is None or ts <= t1)]
        if not rows:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        busy = [r for r in rows if (num(r[3]) or 0) >= 50] or rows
        sm = [num(r[0]) for r in busy if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in busy for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(busy)}


# -------------------------------------------------------------------- timing

KERNEL_TIMING = ("per-launch CUDA events on the launch stream, over a second timed pass of the "
                 "same K steps (the step time is taken without them)")


def _flush(buf):
    buf.add_(1)


def time_steps(fn, steps, warmup, flush_buf, stream, barrier):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    # one extra flush queued ahead: the first timed step's launches are
    # enqueued while the GPU is still busy, as those of every later step are
    _flush(flush_buf)
    evs = []
    for _ in range(steps):
        _flush(flush_buf)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_e2e(r, steps, warmup, stream, barrier):
    """Mean ms per step of K pipelined end-to-end steps: from an event before the
    first input copy to one after the last output has been read back.  No L2
    flush between steps (it would sit inside the timed span): every workload's
    step touches more than L2 holds (its states or its workspace), and inputs
    just copied in are where a serving loop finds them."""
    import torch
    for _ in range(warmup):
        r.e2e_step(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    r.s_in.wait_stream(stream)   # the first copy starts after the start event
    for _ in range(steps):
        r.e2e_step(stream)
    stream.wait_stream(r.s_out)  # the end event follows the last read-back
    b.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def cpu_baseline(key, case, runs=3):
    """The oracle's float build (the same C source as the parity oracle, built with
    float arithmetic, OpenMP over tokens and over (sequence, value head)) timed on
    the whole workload: the median of `runs` runs on all host cores."""
    import oracle
    od = oracle.Dims(case.n_k_heads, case.n_v_heads, case.d_k, case.d_v, case.conv_k, case.act)
    times = []
    for _ in range(runs):
        t0 = time.perf_counter()
        oracle.gdn_f32(od, case.cu_seqlens, case.x, case.z, case.a, case.b, case.conv_w,
                       case.A_log, case.dt_bias, case.norm_w, case.conv_state, case.state)
        times.append(time.perf_counter() - t0)
    med = statistics.median(times)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"the whole workload ({case.n_seq} sequences, {case.n_tokens} tokens, all "
              f"{case.n_v_heads} heads): the oracle's C source built with float arithmetic, "
              f"OpenMP over tokens and over (sequence, value head), median of {runs} runs")
    return {"value": case.n_tokens / med, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample, "seconds_per_run": med}


def h2d_ceiling(nbytes, device, reps=10):
    """GB/s of a plain pinned host-to-device copy of `nbytes` (the ceiling of the
    end-to-end figure when the step's input copy bounds it)."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        dst.copy_(src, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return nbytes * reps / (a.elapsed_time(b) / 1e3) / 1e9


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import gated_deltanet_linear_mixer_gb300 as gdn
    from gated_deltanet_linear_mixer_gb300 import _build, workloads
    from gated_deltanet_linear_mixer_gb300.sharding import max_over_ranks

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)

    def barrier():
        if world > 1:
            dist.barrier()

    if rank == 0 or world == 1:
        _build.build()
    barrier()
    gdn.load()
    peaks = _peaks()
    stream = torch.cuda.current_stream(device)
    flush_buf = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    sampler = ClockSampler(index=local)
    sampler.start()

    keys = ["prefill"] + [k for k in ("decode", "varlen", "spec_verify", "spec_replay", "layer",
                                      "kda_prefill") if k in args.extras]
    results = {}
    total_launches = 0
    for key in keys:
        case = workloads.config(WORKLOADS[key])
        if key == "kda_prefill":
            case = workloads.with_per_channel_decay(case, KDA_SEED)
        r = Runner(key, case, device)
        r.step()  # one untimed call: one-time costs (module loading, library setup) stay out
        torch.cuda.synchronize()
        t_start = time.time()
        # the step time, without per-launch instrumentation (the library's
        # timing events between launches cost a few microseconds each)
        ms = time_steps(r.step, args.steps, args.warmup, flush_buf, stream, barrier)
        # the same K steps again with a CUDA event pair around every launch,
        # recorded on its stream: per-kernel durations for the roofline
        gdn.timing_enable(True)
        time_steps(r.step, args.steps, args.warmup, flush_buf, stream, barrier)
        rep = gdn.timing_report()
        gdn.timing_enable(False)
        t_stop = time.time()
        # timing_report counts warm-up launches too: scale to the timed steps
        per_step_launch = {k: v[0] / (args.steps + args.warmup) for k, v in rep.items()}
        launches = int(round(sum(per_step_launch.values()) * args.steps))
        mean_ms = statistics.mean(ms)
        t_max = max_over_ranks(mean_ms, device=device)
        tok_s = world * r.tokens / (t_max / 1e3)
        # dominant kernel: largest total time
        dom = max(rep.items(), key=lambda kv: kv[1][1])
        dom_name, (dom_n, dom_ms) = dom
        dom_avg_ms = dom_ms / dom_n
        kb = r.kernel_bytes(dom_name, rep.keys())
        share = dom_ms / sum(v[1] for v in rep.values())
        if dom_name in ("chunk_fused", "chunk_prep_kda", "chunk_scan_kda"):
            # the chunked form's tensor-core contractions (all of them in the
            # fused launch, a kernel's share in the per-channel form's two):
            # measured against the bf16 tensor peak
            fl = r.useful_flops(with_proj=False) if dom_name == "chunk_fused" else r.kernel_flops(dom_name)
            achieved = fl / (dom_avg_ms / 1e3) / 1e12
            roof = {"bound": "tensor", "kernel": dom_name, "achieved": achieved,
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"],
                    "traffic": TRAFFIC.get((r.key, dom_name), (None, None))[0],
                    "traffic_source": TRAFFIC.get((r.key, dom_name), (None, None))[1],
                    "peak_source": peaks["source"] + " (bf16 burst)",
                    "useful_flops_per_launch": fl, "kernel_ms": dom_avg_ms, "kernel_share": share,
                    "kernel_timing": KERNEL_TIMING}
        else:
            achieved = kb / (dom_avg_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "traffic": TRAFFIC.get((r.key, dom_name), (None, None))[0],
                    "traffic_source": TRAFFIC.get((r.key, dom_name), (None, None))[1],
                    "peak_source": peaks["source"],
                    "algorithmic_bytes_per_launch": kb, "kernel_ms": dom_avg_ms,
                    "kernel_share": share, "kernel_timing": KERNEL_TIMING}
        step_bytes = r.algorithmic_bytes()
        res = {
            "value": tok_s, "unit": UNIT, "ms_per_step": t_max,
            "config": {"workload": case.name, "n_seq": case.n_seq, "tokens": r.tokens,
                       "Hk": case.n_k_heads, "Hv": case.n_v_heads, "d_k": case.d_k,
                       "d_v": case.d_v, "K": case.conv_k, "act": case.act,
                       "l2": "256 MiB buffer written between timed steps"},
            "roofline": roof,
            "step_hbm": {"algorithmic_bytes": step_bytes,
                         "achieved_gbs": step_bytes / (t_max / 1e3) / 1e9,
                         "frac": step_bytes / (t_max / 1e3) / 1e9 / peaks["hbm_gbs"]},
            "kernels": {k: {"launches_per_step": per_step_launch[k], "ms_per_launch": v[1] / v[0]}
                        for k, v in rep.items()},
            "gpu_launches": launches,
            "clocks": sampler.summary(t_start, t_stop),
        }
        if case.mode == "prefill":
            fl = r.useful_flops()
            res["roofline_tensor"] = {
                "useful_flops_per_step": fl, "chunk": 64,
                "achieved_tflops": fl / (t_max / 1e3) / 1e12,
                "peak": peaks["bf16_tflops"],
                "frac": fl / (t_max / 1e3) / 1e12 / peaks["bf16_tflops"]}
        # end to end through the public API with host buffers
        r.setup_e2e()
        e2e_mean = max_over_ranks(time_e2e(r, args.steps, args.warmup, stream, barrier), device=device)
        res["e2e"] = {"value": world * r.tokens / (e2e_mean / 1e3), "unit": UNIT,
                      "h2d_bytes_per_step": r.h2d, "d2h_bytes_per_step": r.d2h,
                      "ms_per_step": e2e_mean,
                      "pipelining": "H2D of step i+1 and D2H of step i-1 on two copy streams "
                                    "while step i computes",
                      "l2": "no flush between steps: each step touches more than L2 holds"}
        if r.h2d >= (16 << 20):  # where the input copy can bound the step: its ceiling beside it
            gbs = h2d_ceiling(r.h2d, device)
            res["e2e"]["h2d_ceiling_gbs"] = gbs
            res["e2e"]["h2d_bound_tokens_s"] = world * r.tokens / (r.h2d / (gbs * 1e9))
        if rank == 0 and not args.no_cpu_baseline and key in ("prefill", "decode"):
            res["cpu_baseline"] = cpu_baseline(key, case)
        results[key] = res
        total_launches += launches
        del r
        torch.cuda.empty_cache()
    sampler.stop()

    head = results["prefill"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": dict(head["config"], parallelism="replicas" if world > 1 else "single",
                       compute="bf16 activations, fp32 state and accumulation"),
        "roofline": head["roofline"],
        "roofline_tensor": head.get("roofline_tensor"),
        "step_hbm": head["step_hbm"],
        "cpu_baseline": head.get("cpu_baseline"),
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "kernels": head["kernels"],
        "clocks": head["clocks"] or sampler.summary(),
    }
    for k in keys[1:]:
        line[k] = results[k]
    # compact per-workload figures, last in the line (a reader that keeps only
    # the line's tail still has them)
    line["summary"] = {k: {"tokens_s": round(v["value"]), "ms": round(v["ms_per_step"], 4),
                           "kernel": v["roofline"]["kernel"], "bound": v["roofline"]["bound"],
                           "frac": round(v["roofline"]["frac"], 4),
                           "e2e_tokens_s": round(v["e2e"]["value"])}
                       for k, v in results.items()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle (its float build, as cpu_baseline times it) as the reference
    arm, on the prefill workload's config; each step is one whole-workload run."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gated_deltanet_linear_mixer_gb300 import workloads
    import oracle
    case = workloads.config(1)
    od = oracle.Dims(case.n_k_heads, case.n_v_heads, case.d_k, case.d_v, case.conv_k, case.act)
    run = lambda: oracle.gdn_f32(od, case.cu_seqlens, case.x, case.z, case.a, case.b,  # noqa: E731
                                 case.conv_w, case.A_log, case.dt_bias, case.norm_w)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    mean_s = statistics.mean(times)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    v = case.n_tokens / mean_s
    sample = (f"the whole workload per step ({case.n_tokens} tokens, all {case.n_v_heads} heads): "
              "the oracle's C source built with float arithmetic, OpenMP over tokens and over "
              "(sequence, value head)")
    # n_gpus is the launch's N, as in the device arm's line; the oracle itself runs
    # on rank 0's host cores and uses no GPU
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "runs_on": "host cores of rank 0 (no GPU)",
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": case.name, "n_seq": case.n_seq, "tokens": case.n_tokens,
                       "Hk": case.n_k_heads, "Hv": case.n_v_heads, "d_k": case.d_k,
                       "d_v": case.d_v, "K": case.conv_k, "act": case.act},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """One warm-up call and one profiled call of a workload, untimed (for ncu)."""
    import torch
    import gated_deltanet_linear_mixer_gb300 as gdn
    from gated_deltanet_linear_mixer_gb300 import _build, workloads
    _build.build()
    gdn.load()
    key = args.profile
    if key == "decode64":  # a 64-sequence decode step: 128 MiB of state (> L2)
        case = workloads.generate("decode_N64_T1_Hk16_Hv32_d128_bf16", n_k_heads=16, n_v_heads=32,
                                  d_k=128, d_v=128, mode="decode", n_seq=64, tokens_per_seq=1,
                                  dtype="bf16", act="sigmoid", seed=2, state_std=0.05,
                                  conv_state_std=1.0)
        key = "decode"
    elif key == "varlen_small":  # 16 sequences of 128..1024 tokens: the two-kernel launch, ~1 GB
        case = workloads.generate("varlen_small_N16_U128_1024_Hk16_Hv32_d128_bf16", n_k_heads=16,
                                  n_v_heads=32, d_k=128, d_v=128, conv_k=4,
                                  random_lengths=(16, 128, 1024), dtype="bf16", act="silu", seed=3,
                                  state_std=0.05)
        key = "varlen"
    else:
        case = workloads.config(WORKLOADS[key])
        if key == "kda_prefill":
            case = workloads.with_per_channel_decay(case, KDA_SEED)
    r = Runner(key, case, torch.device("cuda", 0))
    for _ in range(2):
        r.step()
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "workload": case.name, "n_seq": case.n_seq,
                      "tokens": int(case.cu_seqlens[-1]) if case.cu_seqlens is not None else None,
                      "device_error": gdn.device_error()}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--extras", default="decode,varlen,spec_verify,spec_replay,layer,kda_prefill",
                    help="comma list of extra workloads in the same line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=sorted(WORKLOADS) + ["decode64", "varlen_small"],
                    help="run one warm-up and one call of a workload, untimed (for ncu)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    args.extras = [e for e in args.extras.split(",") if e]
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
