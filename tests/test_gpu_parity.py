"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Every comparison is element by element on the same seeded inputs, with the
error metric max|gpu - ref| / rms(ref) and the tolerances 1e-4 (fp32
activations) and 2e-2 (bf16 activations, fp32 state).
"""
import copy
import os

import numpy as np
import pytest
import torch

import gated_deltanet_linear_mixer_gb300 as gdn
import oracle
from gated_deltanet_linear_mixer_gb300 import workloads
from gdn_cases import TOL, dims, gpu_decode, gpu_prefill, rel_err, run_oracle, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_deltanet_linear_mixer_gb300 import _build
    _build.build()
    gdn.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _gen(name, **kw):
    base = dict(n_k_heads=2, n_v_heads=4, d_k=128, d_v=128, conv_k=4, dtype="bf16", act="silu",
                seed=11)
    base.update(kw)
    return workloads.generate(name, **base)


def _subcase(case, seqs):
    """The same workload restricted to some sequences (they are independent)."""
    c = copy.copy(case)
    cu = case.cu_seqlens
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seqs]).astype(np.int64)
    lens = [int(cu[i + 1] - cu[i]) for i in seqs]
    c.cu_seqlens = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    c.x, c.z, c.a, c.b = case.x[rows], case.z[rows], case.a[rows], case.b[rows]
    c.state = None if case.state is None else case.state[list(seqs)]
    c.conv_state = None if case.conv_state is None else case.conv_state[list(seqs)]
    return c, rows


PREFILL_CASES = {
    "tiny_fp32": lambda: workloads.config(0),
    "tiny_fp32_slow_decay": lambda: workloads.config(0, slow_decay=True),
    "ragged_bf16_d128_states": lambda: _gen("r1", lengths=[1, 0, 2, 3, 130, 77, 64],
                                            state_std=0.05, conv_state_std=1.0),
    "ragged_f32_dk64_dv128_sigmoid": lambda: _gen("r2", d_k=64, d_v=128, dtype="f32",
                                                  act="sigmoid", lengths=[5, 64, 129, 1],
                                                  state_std=0.05, conv_state_std=1.0, seed=12),
    "bf16_dk128_dv32_K3": lambda: _gen("r3", d_k=128, d_v=32, conv_k=3, lengths=[40, 200],
                                       seed=13, conv_state_std=1.0),
    "bf16_dk32_dv64_K2_gqa4": lambda: _gen("r4", n_k_heads=1, n_v_heads=4, d_k=32, d_v=64,
                                           conv_k=2, lengths=[33, 65], seed=14, state_std=0.1),
    "bf16_slow_decay_long": lambda: _gen("r5", lengths=[700, 333], state_std=0.05, seed=15,
                                         slow_decay=True),
    "f32_slow_decay": lambda: _gen("r6", dtype="f32", lengths=[300, 17], state_std=0.05,
                                   conv_state_std=1.0, seed=16, slow_decay=True),
    # tensor-core path (bf16, d_k = d_v = 128): GQA ratios 1, 2, 3, 4, 8, ragged chunks
    "tc_mha_R1": lambda: _gen("t1", n_k_heads=2, n_v_heads=2, lengths=[150, 64, 65],
                              state_std=0.05, conv_state_std=1.0, seed=31, act="sigmoid"),
    "tc_gqa_R4": lambda: _gen("t2", n_k_heads=1, n_v_heads=4, lengths=[200, 1, 127],
                              state_std=0.05, seed=32),
    "tc_gqa_R3": lambda: _gen("t5", n_k_heads=1, n_v_heads=3, lengths=[96, 64, 33],
                              state_std=0.05, conv_state_std=1.0, seed=35),
    "tc_gqa_R8": lambda: _gen("t6", n_k_heads=1, n_v_heads=8, lengths=[129, 7],
                              state_std=0.05, seed=36, act="sigmoid"),
    "tc_many_short": lambda: _gen("t3", n_k_heads=2, n_v_heads=4,
                                  lengths=[1, 2, 3, 4, 5, 63, 64, 65, 0, 7, 130, 31],
                                  state_std=0.05, conv_state_std=1.0, seed=33),
    "tc_slow_decay_g0": lambda: _gen("t4", n_k_heads=2, n_v_heads=4, lengths=[1000],
                                     state_std=0.05, seed=34, slow_decay=True),
}


@pytest.fixture(autouse=True)
def _no_device_error():
    """Every test must leave the library's sticky device error word at 0."""
    gdn.device_error(reset=True)
    yield
    assert gdn.device_error(reset=True) == 0, "a bounded device wait gave up"


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_prefill_matches_oracle(name):
    case = PREFILL_CASES[name]()
    ref = run_oracle(case)
    got = gpu_prefill(case)
    tol = TOL[case.dtype]
    assert rel_err(got["out"], ref["out"]) <= tol
    assert rel_err(got["state"], ref["state"]) <= tol
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0  # a copy of raw inputs


@pytest.mark.parametrize("name", ["ragged_bf16_d128_states", "ragged_f32_dk64_dv128_sigmoid"])
def test_prefill_in_place_states(name):
    case = PREFILL_CASES[name]()
    ref = run_oracle(case)
    got = gpu_prefill(case, in_place=True)
    tol = TOL[case.dtype]
    assert rel_err(got["out"], ref["out"]) <= tol
    assert rel_err(got["state"], ref["state"]) <= tol
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


POISON_CASES = ["ragged_bf16_d128_states", "tc_many_short", "tc_gqa_R3", "tc_mha_R1",
                "bf16_slow_decay_long"]


@pytest.mark.parametrize("mode", ["fused", "two_kernel", "per_channel"])
@pytest.mark.parametrize("name", POISON_CASES)
def test_prefill_ignores_stale_workspace(name, mode, monkeypatch):
    """A workspace whose every byte is 0xFF (NaN in bf16 and fp32, -1 in the
    chunk table and the item flags) gives the oracle's results on the fused
    launch, the two-kernel launch and the per-channel decay form: nothing in it
    is read before this call writes it, and no padding row or masked tile entry
    reaches an output (a NaN there would survive a multiply by zero)."""
    monkeypatch.setenv("GDN_PREFILL_FUSED", "0" if mode == "two_kernel" else "1")
    case = PREFILL_CASES[name]()
    if mode == "per_channel":
        case = _per_channel(case, seed=95)
    ref = run_oracle(case)
    d, _ = dims(case)
    need = gdn.prefill_workspace_size(d, case.cu_seqlens)
    assert need > 0  # the chunked tensor-core path
    ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")
    gdn.timing_enable(True)
    try:
        got = gpu_prefill(case, workspace=ws)
        names = gdn.timing_report()
    finally:
        gdn.timing_enable(False)
    want = {"fused": "chunk_fused", "two_kernel": "chunk_scan", "per_channel": "chunk_scan_kda"}[mode]
    assert want in names, names
    tol = TOL[case.dtype]
    assert rel_err(got["out"], ref["out"]) <= tol
    assert rel_err(got["state"], ref["state"]) <= tol
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_prefill_without_optional_states():
    """NULL initial state / conv state in, no outputs for them: out still matches."""
    case = _gen("r7", lengths=[50, 3], seed=17)
    ref = run_oracle(case)
    d, _ = dims(case)
    t = upload(case)
    out = gdn.prefill(d, t["params"], case.cu_seqlens, t["x"], t["z"], t["a"], t["b"])
    torch.cuda.synchronize()
    assert rel_err(out, ref["out"]) <= TOL["bf16"]


def test_prefill_zero_sequences_and_empty():
    d, _ = dims(_gen("e", lengths=[1]))
    case = _gen("e", lengths=[0, 0])
    t = upload(case)
    st = torch.full((2, 4, 128, 128), float("nan"), device="cuda")
    gdn.prefill(d, t["params"], [0, 0, 0], t["x"], t["z"], t["a"], t["b"], final_state=st)
    torch.cuda.synchronize()
    assert torch.all(st == 0)   # empty sequences: final state = (zero) initial state


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (32, 128)])
def test_conv_prologue_matches_oracle_stages(dtype, dk, dv):
    case = _gen("c", d_k=dk, d_v=dv, dtype=dtype, lengths=[1, 2, 70, 0, 129, 5],
                conv_state_std=1.0, seed=18)
    ref = run_oracle(case, want_stages=True)
    d, _ = dims(case)
    t = upload(case)
    cs_out = torch.full_like(t["conv_state"], float("nan"))
    qkv, g, beta = gdn.conv(d, t["params"], case.cu_seqlens, t["x"], t["a"], t["b"],
                            conv_state_in=t["conv_state"], conv_state_out=cs_out)
    torch.cuda.synchronize()
    kd = d.n_k_heads * dk
    tol = TOL[dtype]
    tt = case.n_tokens
    assert rel_err(qkv[:, :kd], ref["q_hat"].reshape(tt, -1)) <= tol
    assert rel_err(qkv[:, kd:2 * kd], ref["k_hat"].reshape(tt, -1)) <= tol
    assert rel_err(qkv[:, 2 * kd:], ref["v"].reshape(tt, -1)) <= tol
    assert rel_err(g, ref["g"]) <= 1e-5
    assert rel_err(beta, ref["beta"]) <= 1e-6
    assert rel_err(cs_out, ref["conv_state"]) == 0.0


DECODE_CASES = {
    "bf16_T1_sigmoid": lambda: _gen("d1", mode="decode", n_seq=6, tokens_per_seq=1,
                                    act="sigmoid", state_std=0.05, conv_state_std=1.0, seed=21),
    "bf16_T4_inter": lambda: _gen("d2", mode="decode", n_seq=5, tokens_per_seq=4,
                                  act="sigmoid", state_std=0.05, conv_state_std=1.0, seed=22,
                                  want_inter=True),
    "f32_T3_silu_dk64": lambda: _gen("d3", mode="decode", n_seq=3, tokens_per_seq=3, d_k=64,
                                     dtype="f32", state_std=0.05, conv_state_std=1.0, seed=23),
    "bf16_T16_max": lambda: _gen("d4", mode="decode", n_seq=2, tokens_per_seq=16,
                                 act="sigmoid", state_std=0.05, conv_state_std=1.0, seed=24,
                                 want_inter=True),
    "f32_T2_slow_decay": lambda: _gen("d5", mode="decode", n_seq=4, tokens_per_seq=2,
                                      dtype="f32", state_std=0.05, conv_state_std=1.0, seed=25,
                                      slow_decay=True),
}


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_decode_matches_oracle(name):
    case = DECODE_CASES[name]()
    ref = run_oracle(case, want_inter=case.want_inter)
    got = gpu_decode(case, inter=case.want_inter)
    tol = TOL[case.dtype]
    assert rel_err(got["out"], ref["out"]) <= tol
    if case.want_inter:
        n, tt = case.n_seq, case.tokens_per_seq
        inter_ref = ref["inter"].reshape(n, tt, *ref["inter"].shape[1:])
        assert rel_err(got["inter"], inter_ref) <= tol
        # verify mode: resident state and conv state are read only
        assert rel_err(got["state"], case.state) == 0.0
        assert rel_err(got["conv_state"], case.conv_state) == 0.0
    else:
        assert rel_err(got["state"], ref["state"]) <= tol
        assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_decode_commit_keeps_accepted_prefix():
    case = _gen("cm", mode="decode", n_seq=5, tokens_per_seq=4, act="sigmoid", state_std=0.05,
                conv_state_std=1.0, seed=26, want_inter=True)
    got = gpu_decode(case, inter=True)
    d, _ = dims(case)
    t = upload(case)
    accepted = torch.tensor([0, 1, 2, 3, 4], dtype=torch.int32, device="cuda")
    state = t["state"].clone()
    cs = t["conv_state"].clone()
    gdn.decode_commit(d, accepted, t["x"].view(5, 4, -1), got["inter"], state, cs)
    torch.cuda.synchronize()
    for i, j in enumerate([0, 1, 2, 3, 4]):
        sub, _ = _subcase(case, [i])
        sub.cu_seqlens = np.array([0, j], dtype=np.int32)
        sub.x, sub.z, sub.a, sub.b = sub.x[:j], sub.z[:j], sub.a[:j], sub.b[:j]
        ref = run_oracle(sub)
        assert rel_err(state[i], ref["state"][0]) <= TOL["bf16"]
        assert rel_err(cs[i], ref["conv_state"][0]) == 0.0


@pytest.mark.parametrize("d_k", [128, 64])
def test_verify_then_replay_gives_the_committed_state(d_k, monkeypatch):
    """Rollback by replay: gdn_verify runs the drafts against a read-only state
    (its outputs are gdn_decode's up to rounding, bit for bit on the
    token-by-token path, and nothing else is written); replaying each
    sequence's accepted prefix with gdn_prefill from the kept state and history
    (the token-recurrent path: every prefix is short) gives the state that
    gdn_decode wrote as an intermediate and the history gdn_decode_commit keeps,
    bit for bit, and both match the oracle run on the accepted prefix."""
    n, tt = 6, 4
    accepted = [0, 1, 2, 3, 4, 2]
    case = _gen("rp", mode="decode", n_seq=n, tokens_per_seq=tt, d_k=d_k, act="sigmoid",
                state_std=0.05, conv_state_std=1.0, seed=27, want_inter=True)
    d, _ = dims(case)
    t = upload(case)
    x, z, a, b = (t[k].view(n, tt, -1) for k in ("x", "z", "a", "b"))
    st0, cs0 = t["state"].clone(), t["conv_state"].clone()
    inter = torch.full((n, tt, d.n_v_heads, d.d_k, d.d_v), float("nan"), device="cuda")
    out_ref = gdn.decode(d, t["params"], x, z, a, b, st0.clone(), cs0.clone(), inter)
    st_v, cs_v = st0.clone(), cs0.clone()
    out_v = gdn.verify(d, t["params"], x, z, a, b, st_v, conv_state=cs_v)  # all drafts in one pass
    monkeypatch.setenv("GDN_VERIFY_TOKENWISE", "1")
    out_w = gdn.verify(d, t["params"], x, z, a, b, st_v, conv_state=cs_v)  # token by token
    monkeypatch.delenv("GDN_VERIFY_TOKENWISE")
    torch.cuda.synchronize()
    assert torch.equal(out_w, out_ref)
    assert rel_err(out_v.reshape(n * tt, -1), run_oracle(case)["out"]) <= TOL["bf16"]
    assert torch.equal(st_v, st0) and torch.equal(cs_v, cs0)
    # replay: the accepted prefixes packed as one variable-length prefill
    cu = np.concatenate([[0], np.cumsum(accepted)]).astype(np.int32)
    pick = lambda u: torch.cat([u[i, :j] for i, j in enumerate(accepted)])  # noqa: E731
    st_r, cs_r = st0.clone(), torch.empty_like(cs0)
    gdn.prefill(d, t["params"], cu, pick(x), pick(z), pick(a), pick(b), initial_state=st_r,
                final_state=st_r, conv_state_in=cs0, conv_state_out=cs_r)
    # the commit path on the same intermediates
    st_c, cs_c = st0.clone(), cs0.clone()
    gdn.decode_commit(d, torch.tensor(accepted, dtype=torch.int32, device="cuda"), x, inter,
                      st_c, cs_c)
    torch.cuda.synchronize()
    assert torch.equal(cs_r, cs_c)
    assert torch.equal(st_r, st_c)
    for i, j in enumerate(accepted):
        sub, _ = _subcase(case, [i])
        sub.cu_seqlens = np.array([0, j], dtype=np.int32)
        sub.x, sub.z, sub.a, sub.b = sub.x[:j], sub.z[:j], sub.a[:j], sub.b[:j]
        ref = run_oracle(sub)
        assert rel_err(st_r[i], ref["state"][0]) <= TOL["bf16"]


READ_ONLY_VERIFY_CASES = {
    # d_k, d_v, tokens, conv_k, act, dtype, GQA (Hk, Hv), conv history given
    "d128_T4": (128, 128, 4, 4, "silu", "bf16", (2, 4), True),
    "d128_T3_sigmoid": (128, 128, 3, 4, "sigmoid", "bf16", (1, 3), True),
    "d128_T1_no_history": (128, 128, 1, 4, "silu", "bf16", (2, 2), False),
    "dk64_dv128_T2_K3": (64, 128, 2, 3, "silu", "bf16", (2, 4), True),
    "dk128_dv64_T4_f32": (128, 64, 4, 4, "sigmoid", "f32", (1, 4), True),
    "dk32_dv32_T4_K2": (32, 32, 4, 2, "silu", "bf16", (1, 8), True),
    "dk128_dv32_T3_f32_K3": (128, 32, 3, 3, "silu", "f32", (2, 4), False),
    "d128_T2_f32": (128, 128, 2, 4, "silu", "f32", (2, 4), True),
}


@pytest.mark.parametrize("name", sorted(READ_ONLY_VERIFY_CASES))
def test_read_only_verify_matches_oracle(name):
    """gdn_verify of up to four drafts takes all of them in one pass over the
    state (unrolled form of the token rule): its outputs match the oracle's
    decode of the same tokens, and neither the state nor the history moves."""
    d_k, d_v, tt, k, act, dt, (hk, hv), hist = READ_ONLY_VERIFY_CASES[name]
    n = 5
    case = _gen("ro" + name, mode="decode", n_seq=n, tokens_per_seq=tt, d_k=d_k, d_v=d_v,
                conv_k=k, act=act, dtype=dt, n_k_heads=hk, n_v_heads=hv, state_std=0.05,
                conv_state_std=1.0 if hist else None, seed=41)
    ref = run_oracle(case)
    d, _ = dims(case)
    t = upload(case)
    x, z, a, b = (t[key].view(n, tt, -1) for key in ("x", "z", "a", "b"))
    st = t["state"].clone()
    cs = None if t["conv_state"] is None else t["conv_state"].clone()
    out = gdn.verify(d, t["params"], x, z, a, b, st, conv_state=cs)
    torch.cuda.synchronize()
    assert rel_err(out.reshape(n * tt, -1), ref["out"]) <= TOL[dt]
    assert torch.equal(st, t["state"])
    if cs is not None:
        assert torch.equal(cs, t["conv_state"])


def test_decode_equals_prefill_of_same_tokens():
    """T decode tokens against a state == prefill of those T tokens from that state."""
    case = _gen("dp", mode="decode", n_seq=3, tokens_per_seq=4, state_std=0.05,
                conv_state_std=1.0, seed=27)
    dec = gpu_decode(case)
    pre = gpu_prefill(case)  # bf16, d=128: the tensor-core path
    assert rel_err(dec["out"], pre["out"].float().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(dec["state"], pre["state"].cpu().numpy()) <= TOL["bf16"]
    assert rel_err(dec["conv_state"], pre["conv_state"].float().cpu().numpy()) == 0.0


def test_invalid_arguments_raise():
    case = _gen("iv", lengths=[4])
    d, _ = dims(case)
    t = upload(case)
    with pytest.raises(gdn.GDNError, match="cu_seqlens"):
        gdn.prefill(d, t["params"], torch.tensor([1, 4], dtype=torch.int32), t["x"], t["z"], t["a"], t["b"])
    with pytest.raises(gdn.GDNError, match="T must be"):
        st = torch.zeros((1, 4, 128, 128), device="cuda")
        x = torch.zeros((1, 17, d.conv_dim), dtype=d.dtype, device="cuda")
        gdn.decode(d, t["params"], x, torch.zeros((1, 17, 512), dtype=d.dtype, device="cuda"),
                   torch.zeros((1, 17, 4), dtype=d.dtype, device="cuda"),
                   torch.zeros((1, 17, 4), dtype=d.dtype, device="cuda"), st)


def _with_options(case, head_map="contiguous", decay_form="A_log"):
    """The ABI options of the pages' GGUF checkpoints on a generated case: the
    tiled value-to-key map, and the decay coefficient given instead of A_log
    (rounded to fp32 first, so that both sides read the same values).  A copy:
    the named workloads are cached and shared."""
    case = copy.copy(case)
    case.head_map, case.decay_form = head_map, decay_form
    if decay_form == "coef":
        case.A_log = (-np.exp(case.A_log)).astype(np.float32).astype(np.float64)
    return case


@pytest.mark.parametrize("name,decay_form", [("tc_gqa_R4", "A_log"), ("tc_gqa_R8", "coef"),
                                             ("ragged_bf16_d128_states", "coef"),
                                             ("bf16_dk32_dv64_K2_gqa4", "A_log"),
                                             ("ragged_f32_dk64_dv128_sigmoid", "coef")])
def test_prefill_tiled_head_map_and_decay_coef_match_oracle(name, decay_form):
    """Tensor-core (d=128 bf16) and token-recurrent paths with the tiled map."""
    case = _with_options(PREFILL_CASES[name](), "tiled", decay_form)
    ref = run_oracle(case)
    got = gpu_prefill(case)
    tol = TOL[case.dtype]
    assert rel_err(got["out"], ref["out"]) <= tol
    assert rel_err(got["state"], ref["state"]) <= tol


def test_decode_tiled_head_map_and_decay_coef_match_oracle():
    case = _with_options(_gen("dt", mode="decode", n_seq=5, tokens_per_seq=4, n_k_heads=2,
                              n_v_heads=6, act="sigmoid", state_std=0.05, conv_state_std=1.0,
                              seed=28, want_inter=True), "tiled", "coef")
    ref = run_oracle(case, want_inter=True)
    got = gpu_decode(case, inter=True)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    n, tt = case.n_seq, case.tokens_per_seq
    assert rel_err(got["inter"], ref["inter"].reshape(n, tt, *ref["inter"].shape[1:])) <= TOL["bf16"]


def _per_channel(case, seed):
    """The case with one decay per key channel (a copy; see the workloads module)."""
    return workloads.with_per_channel_decay(case, seed)


@pytest.mark.parametrize("name", ["ragged_bf16_d128_states", "bf16_slow_decay_long",
                                  "f32_slow_decay", "tc_gqa_R8"])
def test_prefill_per_channel_decay_matches_oracle(name):
    """One decay per key channel: the token-recurrent kernel (fp32) and the
    chunked tensor-core path (bf16, d_k = d_v = 128); the kernels that ran are
    checked, then the results against the oracle."""
    case = _per_channel(PREFILL_CASES[name](), seed=91)
    ref = run_oracle(case)
    gdn.timing_enable(True)
    try:
        got = gpu_prefill(case)
        names = gdn.timing_report()
    finally:
        gdn.timing_enable(False)
    if case.dtype == "bf16" and case.d_k == 128 and case.d_v == 128:
        assert "chunk_prep_kda" in names and "chunk_scan_kda" in names and "recurrent" not in names, names
    else:
        assert "recurrent" in names and "chunk_prep_kda" not in names, names
    tol = TOL[case.dtype]
    assert rel_err(got["out"], ref["out"]) <= tol
    assert rel_err(got["state"], ref["state"]) <= tol


KDA_TC_CASES = ["tc_mha_R1", "tc_gqa_R4", "tc_gqa_R3", "tc_many_short", "tc_slow_decay_g0"]


def _chunked_per_channel(case, want_kernels=True):
    """gpu_prefill of a per-channel case, checking that the chunked tensor-core
    kernels of that form ran (not the token-recurrent one)."""
    gdn.timing_enable(True)
    try:
        got = gpu_prefill(case)
        names = gdn.timing_report()
    finally:
        gdn.timing_enable(False)
    if want_kernels:
        assert "chunk_prep_kda" in names and "chunk_scan_kda" in names, names
        assert "recurrent" not in names, names
    return got


@pytest.mark.parametrize("name", KDA_TC_CASES)
def test_chunked_per_channel_decay_matches_oracle(name):
    """Per-channel decay on the chunked tensor-core path (bf16, d_k = d_v = 128):
    GQA ratios 1, 3, 4, ragged and one-token chunks, many short sequences, a
    1000-token slow-decay sequence; outputs, final states and conv history
    against the oracle."""
    case = _per_channel(PREFILL_CASES[name](), seed=94)
    ref = run_oracle(case)
    got = _chunked_per_channel(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_chunked_per_channel_decay_wide_spread():
    """Channel decays that differ by orders of magnitude within a head: a ~ N(0, 3)
    per channel, so per-token log-decays run from ~0 to about -150 and the
    in-chunk sums of the fast channels reach thousands.  The block factors of
    the Gram products stay <= 1 (nothing overflows) and the result meets the
    oracle."""
    case = _gen("kw", n_k_heads=2, n_v_heads=4, lengths=[300, 64, 17], state_std=0.05,
                conv_state_std=1.0, seed=37)
    case = _per_channel(case, seed=96)
    rng = np.random.default_rng(97)
    case.a = workloads.round_bf16(rng.normal(0.0, 3.0, case.a.shape).astype(np.float32)).astype(np.float64)
    ref = run_oracle(case)
    got = _chunked_per_channel(case)
    assert torch.isfinite(got["out"].float()).all() and torch.isfinite(got["state"]).all()
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["tc_gqa_R4", "tc_mha_R1"])
def test_chunked_per_channel_decay_with_checkpoint_options(name):
    """Per-channel decay on the chunked path with the tiled value-to-key map and
    the decay coefficient given directly (the prep and the scan both look up a
    value head's key head, and the prep forms the decays from the coefficient)."""
    case = _per_channel(_with_options(PREFILL_CASES[name](), "tiled", "coef"), seed=99)
    ref = run_oracle(case)
    got = _chunked_per_channel(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]


def test_chunked_per_channel_decay_in_place_states():
    """Final state over the initial one, new conv history over the old one."""
    case = _per_channel(PREFILL_CASES["ragged_bf16_d128_states"](), seed=100)
    ref = run_oracle(case)
    gdn.timing_enable(True)
    try:
        got = gpu_prefill(case, in_place=True)
        names = gdn.timing_report()
    finally:
        gdn.timing_enable(False)
    assert "chunk_prep_kda" in names
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_full_size_chunked_per_channel_decay_T4096():
    """The 4,096-token Qwen3-Next-shaped prefill with one decay per key channel
    (gate inputs a [T, 32 x 128] ~ N(0, 1), dt_bias [32 x 128] ~ N(0, 0.1))."""
    case = _per_channel(workloads.config(1), seed=98)
    ref = run_oracle(case)
    got = _chunked_per_channel(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]


def test_decode_per_channel_decay_matches_oracle():
    case = _per_channel(_gen("dp", mode="decode", n_seq=4, tokens_per_seq=4, act="sigmoid",
                             state_std=0.05, conv_state_std=1.0, seed=29, want_inter=True), seed=92)
    ref = run_oracle(case, want_inter=True)
    got = gpu_decode(case, inter=True)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    n, tt = case.n_seq, case.tokens_per_seq
    assert rel_err(got["inter"], ref["inter"].reshape(n, tt, *ref["inter"].shape[1:])) <= TOL["bf16"]


@pytest.mark.parametrize("options", ["tiled_coef", "per_channel"])
def test_read_only_verify_options_match_oracle(options):
    """gdn_verify with the checkpoint options: the tiled map with the decay
    coefficient (the one-pass kernel takes them), and per-channel decay (which
    it does not: the token-by-token kernel runs the call)."""
    case = _gen("vo", mode="decode", n_seq=5, tokens_per_seq=4, n_k_heads=2, n_v_heads=6,
                act="sigmoid", state_std=0.05, conv_state_std=1.0, seed=30)
    case = _with_options(case, "tiled", "coef") if options == "tiled_coef" else _per_channel(case, 93)
    ref = run_oracle(case)
    d, _ = dims(case)
    t = upload(case)
    n, tt = case.n_seq, case.tokens_per_seq
    x, z, a, b = (t[key].view(n, tt, -1) for key in ("x", "z", "a", "b"))
    st, cs = t["state"].clone(), t["conv_state"].clone()
    out = gdn.verify(d, t["params"], x, z, a, b, st, conv_state=cs)
    torch.cuda.synchronize()
    assert rel_err(out.reshape(n * tt, -1), ref["out"]) <= TOL["bf16"]
    assert torch.equal(st, t["state"]) and torch.equal(cs, t["conv_state"])


TC_CASES = sorted(k for k in PREFILL_CASES if k.startswith("tc_"))


@pytest.mark.parametrize("name", TC_CASES)
def test_prefill_fused_and_two_kernel_launches_agree(name, monkeypatch):
    """Small batches run prep and scan as one launch (scan clusters wait on
    the prep CTAs' per-chunk flags); GDN_PREFILL_FUSED=0 forces the two-kernel
    launch.  The two differ only in how one split product's three terms are
    summed (rounding): each meets the oracle, and their fp32 states agree to
    1e-3 of the state's RMS (a stale or missing chunk row would be far off)."""
    case = PREFILL_CASES[name]()
    monkeypatch.setenv("GDN_PREFILL_FUSED", "0")
    two = gpu_prefill(case)
    monkeypatch.setenv("GDN_PREFILL_FUSED", "1")
    one = gpu_prefill(case)
    ref = run_oracle(case)
    for got in (one, two):
        assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
        assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(one["state"], two["state"].cpu().numpy()) <= 1e-3


def _layer_inputs(case, hidden, seed, exact=False):
    """bf16 hidden states ~N(0,1) and projection weights ~N(0, 1/in_features).

    exact: hidden states are integers in [-4, 4] and every in_proj row has 8
    nonzero weights of +-1/16, so each projection is a multiple of 1/16 below 3
    in magnitude: exact in bf16 and in any fp32 summation order.  The bf16
    rounding of the projections is then no decision at all, and both sides feed
    the core the same values (with dense weights, the GEMM's fp32 sums and the
    oracle's float64 ones round ~0.1% of the values to neighbouring bf16s, and
    the core's final state is that sensitive)."""
    rng = np.random.default_rng(seed)
    vd, hv = case.n_v_heads * case.d_v, case.n_v_heads
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)  # noqa: E731
    shapes = {"w_qkv": (case.conv_dim, hidden), "w_z": (vd, hidden), "w_a": (hv, hidden),
              "w_b": (hv, hidden), "w_out": (hidden, vd)}
    if not exact:
        h = bf(rng.normal(size=(case.n_tokens, hidden)))
        w = {k: bf(rng.normal(0, 1 / np.sqrt(s[1]), size=s)) for k, s in shapes.items()}
        return h, w
    h = bf(rng.integers(-4, 5, size=(case.n_tokens, hidden)).astype(np.float64))
    w = {}
    for k, (rows, cols) in shapes.items():
        if k == "w_out":  # out_proj rounds nothing on the way: dense
            w[k] = bf(rng.normal(0, 1 / np.sqrt(cols), size=(rows, cols)))
            continue
        m = np.zeros((rows, cols))
        for r in range(rows):
            m[r, rng.choice(cols, 8, replace=False)] = rng.choice([-1 / 16, 1 / 16], 8)
        w[k] = bf(m)
    return h, w


def _layer_check(case, hidden, seed, exact=False, poison=False):
    d, od = dims(case)
    t = upload(case)
    h, w = _layer_inputs(case, hidden, seed, exact)
    proj = gdn.Proj(*(w[k].cuda() for k in ("w_qkv", "w_z", "w_a", "w_b", "w_out")))
    n = case.n_seq
    st = torch.full((n, d.n_v_heads, d.d_k, d.d_v), float("nan"), device="cuda")
    cs = torch.full((n, d.conv_dim, d.conv_k - 1), float("nan"), dtype=d.dtype, device="cuda")
    out = torch.full((case.n_tokens, hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = None
    if poison:  # every byte 0xFF: NaN in the bf16/fp32 intermediates, -1 in the tables
        need = gdn.layer_prefill_workspace_size(d, hidden, case.cu_seqlens)
        ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")
    got = gdn.layer_prefill(d, t["params"], proj, case.cu_seqlens, h.cuda(),
                            initial_state=t["state"], final_state=st,
                            conv_state_in=t["conv_state"], conv_state_out=cs, out=out,
                            workspace=ws)
    torch.cuda.synchronize()
    f = lambda u: u.float().numpy()  # noqa: E731
    ref = oracle.layer(od, case.cu_seqlens, f(h), f(w["w_qkv"]), f(w["w_z"]), f(w["w_a"]),
                       f(w["w_b"]), f(w["w_out"]), case.conv_w, case.A_log, case.dt_bias,
                       case.norm_w, case.conv_state, case.state)
    assert rel_err(got, ref["h_out"]) <= TOL["bf16"]
    assert rel_err(st, ref["state"]) <= TOL["bf16"]
    assert rel_err(cs, ref["conv_state"]) <= TOL["bf16"]


@pytest.mark.parametrize("lengths", [[150, 70, 1], [5, 9, 16]])
def test_layer_prefill_matches_oracle(lengths):
    """in_proj (the tcgen05 GEMM) -> core -> out_proj against the oracle's float64
    projections; [5, 9, 16] takes the short-sequence (token-recurrent) core."""
    case = _gen("ly", lengths=lengths, state_std=0.05, conv_state_std=1.0, seed=41)
    _layer_check(case, hidden=256, seed=141)


@pytest.mark.parametrize("lengths", [[150, 70, 1], [5, 9, 16]])
def test_layer_prefill_ignores_stale_workspace(lengths):
    """The layer from a workspace of 0xFF bytes: the projections' outputs, the
    core's workspace and the gated-norm rows are all written before they are
    read, on the tensor-core and the token-recurrent core."""
    case = _gen("ly", lengths=lengths, state_std=0.05, conv_state_std=1.0, seed=43)
    _layer_check(case, hidden=256, seed=143, poison=True)


def test_layer_prefill_qwen3_next_width():
    """The layer at the workload's head geometry (Hk=16, Hv=32, d=128) and a
    2048-wide model, one 1024-token sequence (the fused tensor-core core), with
    projections exact in bf16 (see _layer_inputs)."""
    case = _gen("lw", n_k_heads=16, n_v_heads=32, lengths=[1024], seed=42)
    _layer_check(case, hidden=2048, seed=142, exact=True)


# ---------------------------------------------------------------- full sizes

@pytest.fixture
def _release_memory():
    """The maximum-size tests hold 20-110 GB; hand it back to the device after
    each, so that the tests after them see the memory free."""
    yield
    torch.cuda.empty_cache()


def test_full_size_prefill_T4096():
    case = workloads.config(1)
    ref = run_oracle(case)
    got = gpu_prefill(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]


@pytest.mark.usefixtures("_release_memory")
@pytest.mark.parametrize("per_channel", [False, True])
def test_max_size_64bit_offsets(per_channel):
    """One 600,000-token sequence, then a 1,000-token one: the second sequence's
    element offsets into x (4.9e9), out (2.5e9) and the workspace's U~ rows
    (2.5e9) pass 2^31, about 70 GB on the device (about 110 GB at the peak with
    per-channel decay). The oracle checks the short sequence (out, final state,
    conv history) and the long one's first 200 outputs (they depend only on its
    first 200 tokens)."""
    free, _ = torch.cuda.mem_get_info()
    if free < (150 if per_channel else 100) * 2 ** 30:
        pytest.skip("not enough free device memory")
    small = _gen("mx", n_k_heads=16, n_v_heads=32, lengths=[200, 1000], state_std=0.05,
                 conv_state_std=1.0, seed=47)
    if per_channel:
        small = _per_channel(small, seed=96)
    ref = run_oracle(small)
    d, _ = dims(small)
    t_small = upload(small)
    long_len = 600000
    total = long_len + 1000
    gen = torch.Generator(device="cuda")
    gen.manual_seed(47)

    def big(name, width):
        v = torch.randn((total, width), generator=gen, device="cuda").to(torch.bfloat16)
        v[:200] = t_small[name][:200]
        v[long_len:] = t_small[name][200:]
        return v

    x = big("x", d.conv_dim)
    z = big("z", d.n_v_heads * d.d_v)
    a = big("a", d.gate_width)
    b = big("b", d.n_v_heads)
    cu = np.array([0, long_len, total], dtype=np.int32)
    st_out = torch.full((2, d.n_v_heads, d.d_k, d.d_v), float("nan"), device="cuda")
    cs_out = torch.full((2, d.conv_dim, d.conv_k - 1), float("nan"), dtype=d.dtype, device="cuda")
    gdn.timing_enable(True)
    try:
        out = gdn.prefill(d, t_small["params"], cu, x, z, a, b, initial_state=t_small["state"],
                          final_state=st_out, conv_state_in=t_small["conv_state"],
                          conv_state_out=cs_out)
        torch.cuda.synchronize()
        names = gdn.timing_report()
    finally:
        gdn.timing_enable(False)
    del x, z, a, b
    # two sequences take the scalar form's two-kernel launch (their 128 scan CTAs
    # leave too few of the 152 slots for a fused prep)
    assert ("chunk_scan_kda" if per_channel else "chunk_scan") in names, names
    assert rel_err(out[long_len:], ref["out"][200:]) <= TOL["bf16"]
    assert rel_err(out[:200], ref["out"][:200]) <= TOL["bf16"]
    assert rel_err(st_out[1], ref["state"][1]) <= TOL["bf16"]
    assert torch.isfinite(st_out[0]).all()
    assert rel_err(cs_out[1], ref["conv_state"][1]) == 0.0


@pytest.mark.usefixtures("_release_memory")
def test_max_size_decode_64bit_state_offsets():
    """One decode step of 20,000 sequences (a 42 GB fp32 state, updated in
    place): the last sequences' state offsets (1.05e10 elements) pass 2^31. The
    oracle checks two sequences at each end of the batch."""
    free, _ = torch.cuda.mem_get_info()
    if free < 80 * 2 ** 30:
        pytest.skip("not enough free device memory")
    small = _gen("md", mode="decode", n_seq=4, tokens_per_seq=1, n_k_heads=16, n_v_heads=32,
                 act="sigmoid", state_std=0.05, conv_state_std=1.0, seed=48)
    ref = run_oracle(small)
    d, _ = dims(small)
    ts = upload(small)
    n = 20000
    pick = [0, 1, n - 2, n - 1]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(48)

    def big(src, shape, std=1.0):
        v = torch.randn(shape, generator=gen, device="cuda")
        v = v.mul_(std) if src.dtype == torch.float32 else v.to(src.dtype)
        v[pick] = src.reshape(4, *shape[1:])
        return v

    vd = d.n_v_heads * d.d_v
    x = big(ts["x"], (n, 1, d.conv_dim))
    z = big(ts["z"], (n, 1, vd))
    a = big(ts["a"], (n, 1, d.gate_width))
    b = big(ts["b"], (n, 1, d.n_v_heads))
    state = big(ts["state"], (n, d.n_v_heads, d.d_k, d.d_v), std=0.05)
    cs = big(ts["conv_state"], (n, d.conv_dim, d.conv_k - 1))
    out = torch.full((n, 1, vd), float("nan"), dtype=d.dtype, device="cuda")
    gdn.decode(d, ts["params"], x, z, a, b, state, cs, None, out)
    torch.cuda.synchronize()
    assert rel_err(out[pick].reshape(4, vd), ref["out"]) <= TOL["bf16"]
    assert rel_err(state[pick], ref["state"]) <= TOL["bf16"]
    assert rel_err(cs[pick], ref["conv_state"]) == 0.0


@pytest.mark.usefixtures("_release_memory")
def test_max_size_verify_64bit_inter_offsets():
    """Speculative verify of 2,048 sequences x 4 drafts writing every
    intermediate state (17 GB): the last sequences' offsets into the
    intermediates (4.3e9 elements) pass 2^31. The oracle checks two sequences at
    each end; the resident state and conv history stay as they were."""
    free, _ = torch.cuda.mem_get_info()
    if free < 60 * 2 ** 30:
        pytest.skip("not enough free device memory")
    small = _gen("mv", mode="decode", n_seq=4, tokens_per_seq=4, n_k_heads=16, n_v_heads=32,
                 act="sigmoid", state_std=0.05, conv_state_std=1.0, seed=49, want_inter=True)
    ref = run_oracle(small, want_inter=True)
    d, _ = dims(small)
    ts = upload(small)
    n, tt = 2048, 4
    pick = [0, 1, n - 2, n - 1]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(49)

    def big(src, shape, std=1.0):
        v = torch.randn(shape, generator=gen, device="cuda")
        v = v.mul_(std) if src.dtype == torch.float32 else v.to(src.dtype)
        v[pick] = src.reshape(4, *shape[1:])
        return v

    vd = d.n_v_heads * d.d_v
    x = big(ts["x"], (n, tt, d.conv_dim))
    z = big(ts["z"], (n, tt, vd))
    a = big(ts["a"], (n, tt, d.gate_width))
    b = big(ts["b"], (n, tt, d.n_v_heads))
    state = big(ts["state"], (n, d.n_v_heads, d.d_k, d.d_v), std=0.05)
    cs = big(ts["conv_state"], (n, d.conv_dim, d.conv_k - 1))
    inter = torch.full((n, tt, d.n_v_heads, d.d_k, d.d_v), float("nan"), device="cuda")
    out = torch.full((n, tt, vd), float("nan"), dtype=d.dtype, device="cuda")
    gdn.decode(d, ts["params"], x, z, a, b, state, cs, inter, out)
    torch.cuda.synchronize()
    assert rel_err(out[pick].reshape(4 * tt, vd), ref["out"]) <= TOL["bf16"]
    inter_ref = ref["inter"].reshape(4, tt, *ref["inter"].shape[1:])
    assert rel_err(inter[pick], inter_ref) <= TOL["bf16"]
    assert rel_err(state[pick], small.state) == 0.0
    assert rel_err(cs[pick], small.conv_state) == 0.0


def test_full_size_prefill_T4096_slow_decay():
    case = workloads.config(1, slow_decay=True)
    ref = run_oracle(case)
    got = gpu_prefill(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]


@pytest.mark.parametrize("kind", ["bf16_tensor_core", "f32_recurrent", "bf16_decode"])
def test_saturated_gates(kind):
    """Gate inputs at the ends of their range, all exact in bf16: a + dt_bias past
    softplus's identity threshold (20) and far below 0 (no decay at all), beta
    saturated at 0 and 1, mixed token by token, so that the chunked form sees
    in-chunk decays from 1 down to e^-480 (underflow) and the recurrence
    alternates between a full write, no write and a wiped state."""
    if kind == "bf16_decode":
        case = _gen("sat_d", mode="decode", n_seq=3, tokens_per_seq=4, act="sigmoid",
                    state_std=0.05, conv_state_std=1.0, seed=71)
    else:
        case = _gen("sat", dtype="bf16" if kind == "bf16_tensor_core" else "f32",
                    lengths=[300, 65, 17], state_std=0.05, seed=72)
    rng = np.random.default_rng(73)
    case.a = rng.choice([-30.0, -8.0, 0.0, 8.0, 25.0, 30.0], size=case.a.shape).astype(case.a.dtype)
    case.b = rng.choice([-30.0, -5.0, 0.0, 5.0, 30.0], size=case.b.shape).astype(case.b.dtype)
    ref = run_oracle(case)
    if kind == "bf16_decode":
        got = gpu_decode(case)
    else:
        got = gpu_prefill(case)
    tol = TOL["f32"] if kind == "f32_recurrent" else TOL["bf16"]
    assert rel_err(got["out"], ref["out"]) <= tol
    assert rel_err(got["state"], ref["state"]) <= tol


def test_decode_at_the_sequence_limit():
    """A decode step of exactly GDN_MAX_SEQUENCES sequences (the largest grid the
    kernels are launched with), small heads so that the state stays small."""
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                             "include", "gdn.h")).read()
    limit = int(text.split("#define GDN_MAX_SEQUENCES")[1].split()[0])
    case = _gen("maxseq", mode="decode", n_seq=limit, tokens_per_seq=1, n_k_heads=1, n_v_heads=1,
                d_k=32, d_v=32, dtype="f32", act="sigmoid", state_std=0.05, conv_state_std=1.0,
                seed=81)
    ref = run_oracle(case)
    got = gpu_decode(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["f32"]
    assert rel_err(got["state"], ref["state"]) <= TOL["f32"]
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_long_single_sequence_fused_launch():
    """One 32,768-token sequence (512 chunks, long-memory gates so that the state
    carries across every chunk) through the fused launch, whose scan waits on
    prep's per-chunk flags 512 times; matches the oracle, and so does the
    two-kernel launch, their fp32 states within 1e-3 of the RMS."""
    case = _gen("long", n_k_heads=2, n_v_heads=4, lengths=[32768], state_std=0.05, seed=61,
                slow_decay=True)
    t = upload(case)
    got = gpu_prefill(case, t)
    ref = run_oracle(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"].float(), ref["conv_state"]) == 0.0
    os.environ["GDN_PREFILL_FUSED"] = "0"
    try:
        two = gpu_prefill(case, t)
    finally:
        del os.environ["GDN_PREFILL_FUSED"]
    assert rel_err(two["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(two["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["state"], two["state"].cpu().numpy()) <= 1e-3
    code = gdn.device_error()
    assert code == 0


@pytest.mark.parametrize("slow", [False, True])
def test_full_size_varlen_prefill_all_sequences(slow):
    """The whole 16-sequence workload (64,523 tokens, two-kernel launch) against
    the oracle, every sequence: output, final state and conv history."""
    case = workloads.config(3, slow_decay=slow)
    got = gpu_prefill(case)
    ref = run_oracle(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"].float(), ref["conv_state"]) == 0.0


def test_full_size_varlen_per_channel_decay():
    """The 16-sequence workload with one decay per key channel: 32,480 (chunk,
    value head) items, about 214 for each of the prep's persistent CTAs, then
    the per-channel scan; every sequence against the oracle."""
    case = _per_channel(workloads.config(3), seed=101)
    got = _chunked_per_channel(case)
    ref = run_oracle(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"].float(), ref["conv_state"]) == 0.0


def test_full_size_decode_256():
    case = workloads.config(2)
    ref = run_oracle(case)
    got = gpu_decode(case)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    assert rel_err(got["state"], ref["state"]) <= TOL["bf16"]
    assert rel_err(got["conv_state"], ref["conv_state"]) == 0.0


def test_read_only_verify_many_items_per_cta():
    """More (sequence, value head) items than resident CTAs, so that each CTA
    walks several items (its next state copy in flight while one computes):
    600 sequences x 4 heads against at most two CTAs per SM."""
    n, tt = 600, 3
    case = _gen("rm", mode="decode", n_seq=n, tokens_per_seq=tt, n_k_heads=2, n_v_heads=4,
                d_k=64, d_v=64, state_std=0.05, conv_state_std=1.0, seed=43)
    ref = run_oracle(case)
    d, _ = dims(case)
    t = upload(case)
    x, z, a, b = (t[key].view(n, tt, -1) for key in ("x", "z", "a", "b"))
    st, cs = t["state"].clone(), t["conv_state"].clone()
    out = gdn.verify(d, t["params"], x, z, a, b, st, conv_state=cs)
    torch.cuda.synchronize()
    assert rel_err(out.reshape(n * tt, -1), ref["out"]) <= TOL["bf16"]
    assert torch.equal(st, t["state"]) and torch.equal(cs, t["conv_state"])


def test_full_size_read_only_verify_64x4():
    """The speculative-verify workload through gdn_verify (one pass over each
    state for all four drafts): outputs against the oracle, state untouched."""
    case = workloads.config(4)
    ref = run_oracle(case)
    d, _ = dims(case)
    t = upload(case)
    n, tt = case.n_seq, case.tokens_per_seq
    x, z, a, b = (t[key].view(n, tt, -1) for key in ("x", "z", "a", "b"))
    st, cs = t["state"].clone(), t["conv_state"].clone()
    out = gdn.verify(d, t["params"], x, z, a, b, st, conv_state=cs)
    torch.cuda.synchronize()
    assert rel_err(out.reshape(n * tt, -1), ref["out"]) <= TOL["bf16"]
    assert torch.equal(st, t["state"]) and torch.equal(cs, t["conv_state"])


def test_full_size_spec_verify_64x4():
    case = workloads.config(4)
    ref = run_oracle(case, want_inter=True)
    got = gpu_decode(case, inter=True)
    assert rel_err(got["out"], ref["out"]) <= TOL["bf16"]
    inter_ref = ref["inter"].reshape(64, 4, 32, 128, 128)
    assert rel_err(got["inter"], inter_ref) <= TOL["bf16"]
