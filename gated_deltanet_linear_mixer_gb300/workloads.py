"""Seeded synthetic inputs for the GDN mixer core.

This module holds no arithmetic of the method: it only draws inputs.  Both the
CUDA path's tests/benchmark and the CPU oracle read the arrays it returns, so
both sides see the same values (bf16 activations are rounded here, once, and the
oracle reads the rounded values).

Recipe (one generator per case, ``numpy.random.default_rng(seed)``, PCG64):
draw order conv_w, A_log, dt_bias, norm_w, lengths (random-length cases only),
initial state, conv state, x, z, a, b.  The small parameters are drawn in
float64; the large arrays (states, x, z, a, b) as float32 standard normals that
are then scaled.  Distributions: x (the pre-conv packed
q|k|v), z, a, b ~ N(0, 1); A_log = log U[1, 16]; dt_bias ~ N(0, 0.1);
conv_w ~ N(0, 0.5) of shape [CD, K]; norm_w ~ 1 + N(0, 0.1); states
~ N(0, state_std).  The second parameter of N(.,.) is the standard deviation.
The "slow decay" variant draws A_log = log U[0.001, 0.01] and a ~ N(-3, 1) so
that exp(g) is about 0.9997 and the state is carried across many chunks.
Small parameters (conv_w, A_log, dt_bias, norm_w) and states are float32;
activations (x, z, a, b, conv state) are float32 or bf16-valued float32.
"""
from __future__ import annotations

import copy
import functools
from dataclasses import dataclass, field

import numpy as np


def round_bf16(a: np.ndarray, inplace: bool = False) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32.

    For finite inputs u + 0x7FFF + lsb stays below 2^32, so uint32 arithmetic is
    exact; non-finite values are left as they are.  Works in row blocks to keep
    temporaries small."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    if not inplace:
        f = f.copy()
    flat = f.reshape(-1)
    step = 1 << 22
    for i in range(0, flat.size, step):
        blk = flat[i:i + step]
        u = blk.view(np.uint32)
        fin = np.isfinite(blk)
        tmp = (u >> np.uint32(16)) & np.uint32(1)
        tmp += np.uint32(0x7FFF)
        r = (u + tmp) & np.uint32(0xFFFF0000)
        u[fin] = r[fin]
    return f


def _normal(rng, mean, std, size):
    """Normal draws made as float32 standard normals (fast), then scaled in place."""
    out = np.empty(size, dtype=np.float32)
    rng.standard_normal(dtype=np.float32, out=out)
    if std != 1.0:
        out *= np.float32(std)
    if mean != 0.0:
        out += np.float32(mean)
    return out


@dataclass
class Case:
    """One synthetic workload: geometry, sequence layout and host arrays."""
    name: str
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    conv_k: int
    dtype: str                 # "f32" or "bf16": activations' storage type
    act: str                   # "silu" or "sigmoid"
    mode: str                  # "prefill" (packed, cu_seqlens) or "decode" (T per sequence)
    cu_seqlens: np.ndarray     # int32 [N+1]
    tokens_per_seq: int | None  # decode only
    want_inter: bool
    x: np.ndarray              # [T_total, CD]
    z: np.ndarray              # [T_total, Hv*dv]
    a: np.ndarray              # [T_total, Hv]
    b: np.ndarray              # [T_total, Hv]
    conv_w: np.ndarray         # [CD, K]
    A_log: np.ndarray          # [Hv]
    dt_bias: np.ndarray        # [Hv]
    norm_w: np.ndarray         # [dv]
    conv_state: np.ndarray | None  # [N, CD, K-1]
    state: np.ndarray | None       # [N, Hv, dk, dv]
    meta: dict = field(default_factory=dict)

    @property
    def n_seq(self) -> int:
        return int(self.cu_seqlens.size - 1)

    @property
    def n_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def conv_dim(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v


def generate(name, *, n_k_heads, n_v_heads, d_k, d_v, conv_k=4, lengths=None,
             n_seq=None, tokens_per_seq=None, random_lengths=None, dtype="bf16",
             act="silu", seed=0, state_std=None, conv_state_std=None,
             slow_decay=False, mode="prefill", want_inter=False) -> Case:
    """Draw one case.

    Prefill: give ``lengths`` (list) or ``random_lengths=(n, lo, hi)`` for
    lengths ~ U{lo..hi}.  Decode: give ``n_seq`` and ``tokens_per_seq``.
    ``state_std``/``conv_state_std`` None means a zero (absent) state.
    """
    rng = np.random.default_rng(seed)
    cd = 2 * n_k_heads * d_k + n_v_heads * d_v
    vd = n_v_heads * d_v
    conv_w = rng.normal(0.0, 0.5, size=(cd, conv_k))
    if slow_decay:
        A_log = np.log(rng.uniform(0.001, 0.01, size=n_v_heads))
    else:
        A_log = np.log(rng.uniform(1.0, 16.0, size=n_v_heads))
    dt_bias = rng.normal(0.0, 0.1, size=n_v_heads)
    norm_w = 1.0 + rng.normal(0.0, 0.1, size=d_v)
    if mode == "decode":
        if n_seq is None or tokens_per_seq is None:
            raise ValueError("decode cases need n_seq and tokens_per_seq")
        lens = np.full(n_seq, tokens_per_seq, dtype=np.int64)
    elif random_lengths is not None:
        cnt, lo, hi = random_lengths
        lens = rng.integers(lo, hi + 1, size=cnt)
    else:
        lens = np.asarray(lengths, dtype=np.int64)
    n = lens.size
    cu = np.zeros(n + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    t = int(cu[-1])
    state = None if state_std is None else _normal(rng, 0.0, state_std, (n, n_v_heads, d_k, d_v))
    conv_state = None
    if conv_state_std is not None:
        conv_state = _normal(rng, 0.0, conv_state_std, (n, cd, conv_k - 1))
    x = _normal(rng, 0.0, 1.0, (t, cd))
    z = _normal(rng, 0.0, 1.0, (t, vd))
    a = _normal(rng, -3.0 if slow_decay else 0.0, 1.0, (t, n_v_heads))
    b = _normal(rng, 0.0, 1.0, (t, n_v_heads))

    def act_cast(arr):
        if arr is None:
            return None
        f = np.ascontiguousarray(arr, dtype=np.float32)
        return round_bf16(f, inplace=True) if dtype == "bf16" else f

    return Case(
        name=name, n_k_heads=n_k_heads, n_v_heads=n_v_heads, d_k=d_k, d_v=d_v, conv_k=conv_k,
        dtype=dtype, act=act, mode=mode, cu_seqlens=cu,
        tokens_per_seq=tokens_per_seq if mode == "decode" else None, want_inter=want_inter,
        x=act_cast(x), z=act_cast(z), a=act_cast(a), b=act_cast(b),
        conv_w=conv_w.astype(np.float32), A_log=A_log.astype(np.float32),
        dt_bias=dt_bias.astype(np.float32), norm_w=norm_w.astype(np.float32),
        conv_state=act_cast(conv_state),
        state=None if state is None else state.astype(np.float32),
        meta={"seed": seed, "slow_decay": slow_decay},
    )


# The five workloads of the Qwen3-Next-shaped GDN layer (Hk=16, Hv=32, dk=dv=128,
# K=4) plus the tiny fp32 case.  Index = seed.
CONFIG_NAMES = [
    "tiny_fp32_prefill_T64_Hk2_Hv4_d32",
    "prefill_T4096_Hk16_Hv32_d128_bf16",
    "decode_N256_T1_Hk16_Hv32_d128_bf16",
    "varlen_prefill_16seq_U128-8192_Hk16_Hv32_d128_bf16",
    "spec_verify_N64_T4_Hk16_Hv32_d128_bf16",
]


@functools.lru_cache(maxsize=4)
def config(i: int, *, slow_decay: bool = False) -> Case:
    """The named workloads (cached per process; treat the arrays as read only).
    ``slow_decay`` swaps in the long-memory gate draw."""
    big = dict(n_k_heads=16, n_v_heads=32, d_k=128, d_v=128, conv_k=4)
    if i == 0:
        return generate(CONFIG_NAMES[0], n_k_heads=2, n_v_heads=4, d_k=32, d_v=32, conv_k=4,
                        lengths=[64], dtype="f32", act="silu", seed=0, slow_decay=slow_decay)
    if i == 1:
        return generate(CONFIG_NAMES[1], lengths=[4096], dtype="bf16", act="silu", seed=1,
                        slow_decay=slow_decay, **big)
    if i == 2:
        return generate(CONFIG_NAMES[2], mode="decode", n_seq=256, tokens_per_seq=1,
                        dtype="bf16", act="sigmoid", seed=2, state_std=0.05,
                        conv_state_std=1.0, slow_decay=slow_decay, **big)
    if i == 3:
        return generate(CONFIG_NAMES[3], random_lengths=(16, 128, 8192), dtype="bf16",
                        act="silu", seed=3, state_std=0.05, slow_decay=slow_decay, **big)
    if i == 4:
        return generate(CONFIG_NAMES[4], mode="decode", n_seq=64, tokens_per_seq=4,
                        dtype="bf16", act="sigmoid", seed=4, state_std=0.05,
                        conv_state_std=1.0, want_inter=True, slow_decay=slow_decay, **big)
    raise ValueError(f"no workload {i}")


def with_per_channel_decay(case: Case, seed: int) -> Case:
    """A copy of `case` with one decay per key channel (the per-channel decayed
    rule): gate inputs a [T, Hv*dk] ~N(0,1) (bf16-rounded for bf16 cases) and
    dt_bias [Hv*dk] ~N(0, 0.1), drawn from `seed`.  A copy because the named
    workloads are cached and shared."""
    c = copy.copy(case)
    rng = np.random.default_rng(seed)
    a = rng.normal(size=(case.a.shape[0], case.n_v_heads * case.d_k))
    c.a = round_bf16(a.astype(np.float32)).astype(np.float64) if case.dtype == "bf16" else a
    c.dt_bias = rng.normal(0, 0.1, case.n_v_heads * case.d_k)
    c.per_channel_decay = True
    c.name = case.name + "_per_channel_decay"
    return c
