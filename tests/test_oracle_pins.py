"""Pins for the CPU oracle: checks against what the definition and mathematics fix.

None of these re-types the oracle's own formula: each compares it with a library
routine, a closed form, an invariant, a hand-worked example or an independently
derived formulation (the chunked WY form in ``oracle/chunked.py``, the explicit
transition-matrix product below).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from gated_deltanet_linear_mixer_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _dims(hk=2, hv=4, dk=8, dv=8, k=4, act="silu"):
    return oracle.Dims(hk, hv, dk, dv, k, act)


def _rng_case(d, lens, seed=0, state=True, conv_state=True, slow=False):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    t = int(cu[-1])
    n = len(lens)
    c = dict(
        cu=cu,
        x=rng.normal(size=(t, d.conv_dim)),
        z=rng.normal(size=(t, d.n_v_heads * d.d_v)),
        a=rng.normal(-3 if slow else 0, 1, size=(t, d.n_v_heads)),
        b=rng.normal(size=(t, d.n_v_heads)),
        conv_w=rng.normal(0, 0.5, size=(d.conv_dim, d.conv_k)),
        A_log=np.log(rng.uniform(0.001, 0.01, d.n_v_heads) if slow else rng.uniform(1, 16, d.n_v_heads)),
        dt_bias=rng.normal(0, 0.1, d.n_v_heads),
        norm_w=1 + rng.normal(0, 0.1, d.d_v),
        conv_state=rng.normal(size=(n, d.conv_dim, d.conv_k - 1)) if conv_state else None,
        state=rng.normal(0, 0.05, size=(n, d.n_v_heads, d.d_k, d.d_v)) if state else None,
    )
    return c


def _unit_rows(rng, t, h, dk):
    k = rng.normal(size=(t, h, dk))
    return k / np.linalg.norm(k, axis=-1, keepdims=True)


# ----------------------------------------------------------------- a1/a2: conv

def test_conv_hand_worked_golden():
    gold = json.load(open(os.path.join(GOLDEN, "conv_hand_k4.json")))
    d = oracle.Dims(1, 1, 1, 0, 4)  # conv_dim = 2*1*1 + 0 = 2 channels; use channel 0
    x = np.zeros((3, 2))
    x[:, 0] = gold["inputs"]["x"]
    w = np.zeros((2, 4))
    w[0] = gold["inputs"]["w"]
    hist = np.zeros((1, 2, 3))
    hist[0, 0] = gold["inputs"]["history"]
    c, cs = oracle.conv(d, [0, 3], x, w, hist)
    pre = np.array(gold["expected"]["pre_activation"])
    silu = pre / (1 + np.exp(-pre))
    np.testing.assert_allclose(c[:, 0], silu, atol=gold["tolerance_abs"], rtol=0)
    np.testing.assert_allclose(cs[0, 0], gold["expected"]["history_after"], atol=1e-15, rtol=0)


@pytest.mark.parametrize("t", [1, 2, 3, 7, 33])
def test_conv_matches_torch_conv1d(t):
    """Zero history: conv == PyTorch depthwise conv1d with K-1 left zero padding."""
    d = _dims()
    rng = np.random.default_rng(t)
    x = rng.normal(size=(t, d.conv_dim))
    w = rng.normal(0, 0.5, size=(d.conv_dim, d.conv_k))
    c, _ = oracle.conv(d, [0, t], x, w, None)
    xt = torch.from_numpy(x.T.copy())[None]  # [1, CD, T]
    wt = torch.from_numpy(w.copy())[:, None, :]  # [CD, 1, K]
    ref = torch.nn.functional.conv1d(xt, wt, padding=d.conv_k - 1, groups=d.conv_dim)[0, :, :t]
    ref = torch.nn.functional.silu(ref).numpy().T
    np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("split", [1, 2, 3, 5, 9])
def test_conv_history_equals_concatenation(split):
    """Running [0,split) then [split,T) with the carried history == running [0,T)."""
    d = _dims()
    rng = np.random.default_rng(split)
    t = 12
    x = rng.normal(size=(t, d.conv_dim))
    w = rng.normal(0, 0.5, size=(d.conv_dim, d.conv_k))
    full, cs_full = oracle.conv(d, [0, t], x, w, None)
    c1, cs1 = oracle.conv(d, [0, split], x[:split], w, None)
    c2, cs2 = oracle.conv(d, [0, t - split], x[split:], w, cs1)
    np.testing.assert_allclose(np.concatenate([c1, c2]), full, rtol=0, atol=0)
    np.testing.assert_array_equal(cs2, cs_full)


@pytest.mark.parametrize("t", [0, 1, 2, 3, 4, 10])
def test_conv_state_is_last_raw_inputs(t):
    """New history == last K-1 raw inputs, oldest first, shifted in from the old one."""
    d = _dims()
    rng = np.random.default_rng(100 + t)
    x = rng.normal(size=(t, d.conv_dim))
    w = rng.normal(size=(d.conv_dim, d.conv_k))
    old = rng.normal(size=(1, d.conv_dim, d.conv_k - 1))
    _, cs = oracle.conv(d, [0, t], x, w, old)
    seq = np.concatenate([old[0].T, x], axis=0)  # [K-1+T, CD], oldest first
    np.testing.assert_array_equal(cs[0], seq[-(d.conv_k - 1):].T)


def test_conv_packed_sequences_are_independent():
    d = _dims()
    rng = np.random.default_rng(7)
    lens = [5, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = rng.normal(size=(int(cu[-1]), d.conv_dim))
    w = rng.normal(size=(d.conv_dim, d.conv_k))
    hist = rng.normal(size=(3, d.conv_dim, d.conv_k - 1))
    c, cs = oracle.conv(d, cu, x, w, hist)
    for i in range(3):
        ci, csi = oracle.conv(d, [0, lens[i]], x[cu[i]:cu[i + 1]], w, hist[i:i + 1])
        np.testing.assert_array_equal(c[cu[i]:cu[i + 1]], ci)
        np.testing.assert_array_equal(cs[i], csi[0])


# --------------------------------------------------------------- a3: normalise

def test_normalize_closed_form_on_axis_vectors():
    d = _dims(hk=2, hv=2, dk=8, dv=4)
    c = np.zeros((2, d.conv_dim))
    key_dim = d.n_k_heads * d.d_k
    c[0, 3] = 2.5                 # q, head 0, lane 3
    c[0, key_dim + d.d_k + 5] = -0.75  # k, head 1, lane 5
    c[1, 0:d.d_k] = 1.0           # q, head 0: all ones
    qh, kh, v = oracle.normalize(d, c)
    eps = d.l2_eps
    assert qh[0, 0, 3] == pytest.approx(2.5 / math.sqrt(2.5 ** 2 + eps) / math.sqrt(d.d_k), rel=1e-15)
    assert kh[0, 1, 5] == pytest.approx(-0.75 / math.sqrt(0.75 ** 2 + eps), rel=1e-15)
    # all-ones q head: every lane 1/sqrt(dk+eps) * dk^-1/2
    np.testing.assert_allclose(qh[1, 0], 1 / math.sqrt(d.d_k + eps) / math.sqrt(d.d_k), rtol=1e-15)
    # zero vectors stay zero (eps keeps the norm finite)
    assert np.all(kh[0, 0] == 0.0) and np.all(qh[0, 1] == 0.0)
    np.testing.assert_array_equal(v, c[:, 2 * key_dim:].reshape(2, d.n_v_heads, d.d_v))


def test_normalize_norms_are_below_one_by_the_eps_factor():
    d = _dims()
    rng = np.random.default_rng(3)
    c = rng.normal(size=(5, d.conv_dim)) * 0.01
    qh, kh, _ = oracle.normalize(d, c)
    key_dim = d.n_k_heads * d.d_k
    kraw = c[:, key_dim:2 * key_dim].reshape(5, d.n_k_heads, d.d_k)
    ss = (kraw ** 2).sum(-1)
    np.testing.assert_allclose((kh ** 2).sum(-1), ss / (ss + d.l2_eps), rtol=1e-13)
    qraw = c[:, :key_dim].reshape(5, d.n_k_heads, d.d_k)
    qs = (qraw ** 2).sum(-1)
    np.testing.assert_allclose((qh ** 2).sum(-1), qs / (qs + d.l2_eps) / d.d_k, rtol=1e-13)


# ------------------------------------------------------------------- a4: gates

def test_gates_special_values():
    d = _dims(hk=1, hv=4)
    a = np.array([[0.0, 30.0, -5.0, 0.3]])
    b = np.array([[0.0, np.inf, -np.inf, 1.0]])
    A_log = np.array([-np.inf, 0.0, np.log(2.0), 1.5])
    dt_bias = np.array([0.0, 0.0, 0.0, 0.2])
    g, beta = oracle.gates(d, a, b, A_log, dt_bias)
    assert g[0, 0] == 0.0                     # A_log = -inf: no decay, exp(g) = 1
    assert beta[0, 0] == 0.5                  # sigmoid(0)
    assert beta[0, 1] == 1.0 and beta[0, 2] == 0.0
    assert g[0, 1] == -30.0                   # softplus is the identity above 20
    assert g[0, 2] == pytest.approx(-2.0 * math.log1p(math.exp(-5.0)), rel=1e-15)
    assert g[0, 3] == pytest.approx(-math.exp(1.5) * math.log(1 + math.exp(0.5)), rel=1e-14)
    assert beta[0, 3] == pytest.approx(1 / (1 + math.exp(-1.0)), rel=1e-15)


def test_gates_match_torch_softplus():
    d = _dims(hk=1, hv=3)
    rng = np.random.default_rng(11)
    a = rng.normal(0, 8, size=(50, 3))
    b = rng.normal(0, 4, size=(50, 3))
    A_log = np.log(rng.uniform(1, 16, 3))
    dt_bias = rng.normal(0, 0.1, 3)
    g, beta = oracle.gates(d, a, b, A_log, dt_bias)
    sp = torch.nn.functional.softplus(torch.from_numpy(a + dt_bias), beta=1, threshold=20).numpy()
    np.testing.assert_allclose(g, -np.exp(A_log) * sp, rtol=1e-13)
    np.testing.assert_allclose(beta, torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-14)


# ------------------------------------------------------------- a5: recurrence

def test_recurrence_hand_worked_golden():
    gold = json.load(open(os.path.join(GOLDEN, "recurrence_hand_dk2.json")))
    inp = gold["inputs"]
    d = oracle.Dims(1, 1, 2, 2, 4)
    q = np.array(inp["q"])[:, None, :]
    k = np.array(inp["k"])[:, None, :]
    v = np.array(inp["v"])[:, None, :]
    g = np.array(inp["g"])[:, None]
    beta = np.array(inp["beta"])[:, None]
    s0 = np.array(inp["s0"])[None, None]
    o, s1, inter = oracle.recurrence(d, [0, 2], q, k, v, g, beta, s0, want_inter=True)
    tol = gold["tolerance_abs"]
    np.testing.assert_allclose(o[:, 0], gold["expected"]["o"], atol=tol, rtol=0)
    np.testing.assert_allclose(inter[:, 0], gold["expected"]["s_after"], atol=tol, rtol=0)
    np.testing.assert_allclose(s1[0, 0], gold["expected"]["s_after"][-1], atol=tol, rtol=0)


def test_recurrence_beta_zero_is_pure_decay():
    d = _dims(hk=2, hv=4, dk=8, dv=6)
    rng = np.random.default_rng(5)
    t = 9
    q = rng.normal(size=(t, 2, 8))
    k = _unit_rows(rng, t, 2, 8)
    v = rng.normal(size=(t, 4, 6))
    g = -rng.uniform(0, 0.5, size=(t, 4))
    beta = np.zeros((t, 4))
    s0 = rng.normal(size=(1, 4, 8, 6))
    o, s1, _ = oracle.recurrence(d, [0, t], q, k, v, g, beta, s0)
    G = np.cumsum(g, axis=0)
    for h in range(4):
        hk = h // 2
        for i in range(t):
            np.testing.assert_allclose(o[i, h], np.exp(G[i, h]) * (s0[0, h].T @ q[i, hk]), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(s1[0, h], np.exp(G[-1, h]) * s0[0, h], rtol=1e-12)


def test_recurrence_orthonormal_keys_retrieve_exactly():
    """g = 0, beta = 1, orthonormal keys written from S = 0; reading with q = k_j returns v_j."""
    dk, dv, m = 8, 5, 6
    d = oracle.Dims(1, 1, dk, dv, 4)
    rng = np.random.default_rng(9)
    basis, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    keys = basis.T[:m]                       # m orthonormal rows
    vals = rng.normal(size=(m, dv))
    order = rng.permutation(m)
    t = 2 * m
    k = np.zeros((t, 1, dk)); q = np.zeros((t, 1, dk)); v = np.zeros((t, 1, dv))
    beta = np.zeros((t, 1)); g = np.zeros((t, 1))
    k[:m, 0] = keys; v[:m, 0] = vals; beta[:m] = 1.0; q[:m, 0] = keys
    k[m:, 0] = keys[order]; q[m:, 0] = keys[order]   # read phase: beta = 0, no write
    o, s1, _ = oracle.recurrence(d, [0, t], q, k, v, g, beta, None)
    np.testing.assert_allclose(o[m:, 0], vals[order], atol=1e-13)
    np.testing.assert_allclose(o[:m, 0], vals, atol=1e-13)  # each write is read back at once
    np.testing.assert_allclose(s1[0, 0], keys.T @ vals, atol=1e-13)


def test_recurrence_delta_invariant_after_full_write():
    """gamma = beta = 1 and unit k: after the write S'^T k = v whatever the prior S."""
    d = _dims(hk=1, hv=2, dk=6, dv=4)
    rng = np.random.default_rng(21)
    t = 7
    q = rng.normal(size=(t, 1, 6)); k = _unit_rows(rng, t, 1, 6); v = rng.normal(size=(t, 2, 4))
    g = np.zeros((t, 2)); beta = np.ones((t, 2))
    s0 = rng.normal(size=(1, 2, 6, 4))
    _, _, inter = oracle.recurrence(d, [0, t], q, k, v, g, beta, s0, want_inter=True)
    for i in range(t):
        for h in range(2):
            np.testing.assert_allclose(inter[i, h].T @ k[i, 0], v[i, h], atol=1e-12)


def test_recurrence_matches_transition_matrix_product():
    """S_t = (I - beta k k^T) e^g S_{t-1} + beta k v^T, built as explicit matrices."""
    d = _dims(hk=2, hv=4, dk=6, dv=5)
    rng = np.random.default_rng(31)
    t = 11
    q = rng.normal(size=(t, 2, 6)); k = _unit_rows(rng, t, 2, 6); v = rng.normal(size=(t, 4, 5))
    g = -rng.uniform(0, 1, size=(t, 4)); beta = rng.uniform(0, 1, size=(t, 4))
    s0 = rng.normal(size=(1, 4, 6, 5))
    o, s1, inter = oracle.recurrence(d, [0, t], q, k, v, g, beta, s0, want_inter=True)
    for h in range(4):
        hk = h // 2
        s = s0[0, h].copy()
        for i in range(t):
            kk = k[i, hk][:, None]
            trans = np.exp(g[i, h]) * (np.eye(6) - beta[i, h] * kk @ kk.T)
            s = trans @ s + beta[i, h] * kk @ v[i, h][None, :]
            np.testing.assert_allclose(inter[i, h], s, rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(o[i, h], s.T @ q[i, hk], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(s1[0, h], s, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("chunk", [4, 8, 16])
@pytest.mark.parametrize("slow", [False, True])
def test_recurrence_equals_independent_chunked_form(chunk, slow):
    d = _dims(hk=2, hv=4, dk=8, dv=6)
    case = _rng_case(d, [37, 16, 1, 23], seed=chunk, slow=slow)
    c, _ = oracle.conv(d, case["cu"], case["x"], case["conv_w"], case["conv_state"])
    qh, kh, v = oracle.normalize(d, c)
    g, beta = oracle.gates(d, case["a"], case["b"], case["A_log"], case["dt_bias"])
    o, s1, _ = oracle.recurrence(d, case["cu"], qh, kh, v, g, beta, case["state"])
    o2, s2 = chunked.recurrence_chunked(case["cu"], qh, kh, v, g, beta, case["state"], chunk=chunk)
    scale = np.sqrt(np.mean(o ** 2))
    assert np.max(np.abs(o - o2)) / scale < 1e-10
    assert np.max(np.abs(s1 - s2)) / np.sqrt(np.mean(s1 ** 2)) < 1e-10


@pytest.mark.parametrize("chunk", [4, 16])
@pytest.mark.parametrize("spread", [1.0, 30.0])
def test_per_channel_recurrence_equals_independent_chunked_form(chunk, spread):
    """One decay per key channel: the token recurrence against the chunked form
    with per-channel pairwise decay factors (oracle/chunked.py), on decays of
    ordinary size and on decays spread over orders of magnitude between the
    channels (per-token log-decays down to -spread)."""
    d = oracle.Dims(2, 4, 8, 6, 4, "silu", per_channel_decay=True)
    rng = np.random.default_rng(int(chunk + spread))
    cu = [0, 37, 53, 54, 77]
    t = cu[-1]
    q = rng.normal(size=(t, 2, 8)); k = _unit_rows(rng, t, 2, 8); v = rng.normal(size=(t, 4, 6))
    g = -spread * rng.uniform(0, 1, size=(t, 4, 8)) ** 3
    beta = rng.uniform(0, 1, size=(t, 4))
    s0 = rng.normal(size=(4, 4, 8, 6))
    o, s1, _ = oracle.recurrence(d, cu, q, k, v, g, beta, s0)
    o2, s2 = chunked.recurrence_chunked(cu, q, k, v, g, beta, s0, chunk=chunk)
    assert np.max(np.abs(o - o2)) / np.sqrt(np.mean(o ** 2)) < 1e-10
    assert np.max(np.abs(s1 - s2)) / np.sqrt(np.mean(s1 ** 2)) < 1e-10


def test_recurrence_is_jointly_linear_in_state_and_values():
    d = _dims(hk=2, hv=4, dk=8, dv=6)
    rng = np.random.default_rng(41)
    t = 13
    q = rng.normal(size=(t, 2, 8)); k = _unit_rows(rng, t, 2, 8); v = rng.normal(size=(t, 4, 6))
    g = -rng.uniform(0, 1, size=(t, 4)); beta = rng.uniform(0, 1, size=(t, 4))
    s0 = rng.normal(size=(1, 4, 8, 6))
    o1, s1, _ = oracle.recurrence(d, [0, t], q, k, v, g, beta, s0)
    o2, s2, _ = oracle.recurrence(d, [0, t], q, k, -2.5 * v, g, beta, -2.5 * s0)
    np.testing.assert_allclose(o2, -2.5 * o1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s2, -2.5 * s1, rtol=1e-12, atol=1e-14)


def test_recurrence_gqa_groups_are_contiguous():
    """Value heads 2h and 2h+1 read key head h: permuting key heads permutes outputs."""
    d = _dims(hk=2, hv=4, dk=6, dv=4)
    rng = np.random.default_rng(51)
    t = 5
    q = rng.normal(size=(t, 2, 6)); k = _unit_rows(rng, t, 2, 6); v = rng.normal(size=(t, 4, 4))
    g = -rng.uniform(0, 1, size=(t, 4)); beta = rng.uniform(0, 1, size=(t, 4))
    o, _, _ = oracle.recurrence(d, [0, t], q, k, v, g, beta, None)
    d1 = oracle.Dims(1, 1, 6, 4, 4)
    for h in range(4):
        oh, _, _ = oracle.recurrence(d1, [0, t], q[:, h // 2:h // 2 + 1], k[:, h // 2:h // 2 + 1],
                                     v[:, h:h + 1], g[:, h:h + 1], beta[:, h:h + 1], None)
        np.testing.assert_array_equal(o[:, h], oh[:, 0])


# ------------------------------------------------------------ a6: gated norm

@pytest.mark.parametrize("act", ["silu", "sigmoid"])
def test_gated_norm_matches_torch_rms_norm(act):
    d = _dims(hk=1, hv=3, dk=4, dv=16, act=act)
    rng = np.random.default_rng(61)
    o = rng.normal(size=(7, 3, 16)); z = rng.normal(size=(7, 3, 16)); w = 1 + rng.normal(0, 0.1, 16)
    y = oracle.gated_norm(d, o, z, w)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), (16,), weight=torch.from_numpy(w), eps=d.rms_eps)
    zt = torch.from_numpy(z)
    ref = ref * (torch.sigmoid(zt) if act == "sigmoid" else torch.nn.functional.silu(zt))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_gated_norm_constant_rows_closed_form():
    d = _dims(hk=1, hv=2, dk=4, dv=8, act="sigmoid")
    o = np.full((1, 2, 8), -0.3)
    z = np.zeros((1, 2, 8))
    w = np.linspace(0.5, 1.5, 8)
    y = oracle.gated_norm(d, o, z, w)
    expect = -w * 0.5 / math.sqrt(1 + d.rms_eps / 0.09)
    np.testing.assert_allclose(y[0, 0], expect, rtol=1e-14)
    d2 = _dims(hk=1, hv=2, dk=4, dv=8, act="silu")
    np.testing.assert_array_equal(oracle.gated_norm(d2, o, z, w), 0.0)  # silu(0) = 0


# --------------------------------------------------------- composition / modes

def test_gdn_equals_composition_of_stages():
    d = _dims(act="sigmoid")
    case = _rng_case(d, [10, 3], seed=71)
    r = oracle.gdn(d, case["cu"], case["x"], case["z"], case["a"], case["b"], case["conv_w"],
                   case["A_log"], case["dt_bias"], case["norm_w"], case["conv_state"],
                   case["state"], want_inter=True, want_stages=True)
    c, cs = oracle.conv(d, case["cu"], case["x"], case["conv_w"], case["conv_state"])
    qh, kh, v = oracle.normalize(d, c)
    g, beta = oracle.gates(d, case["a"], case["b"], case["A_log"], case["dt_bias"])
    o, s1, inter = oracle.recurrence(d, case["cu"], qh, kh, v, g, beta, case["state"], True)
    y = oracle.gated_norm(d, o, case["z"].reshape(o.shape), case["norm_w"])
    np.testing.assert_array_equal(r["out"], y.reshape(r["out"].shape))
    np.testing.assert_array_equal(r["state"], s1)
    np.testing.assert_array_equal(r["inter"], inter)
    np.testing.assert_array_equal(r["conv_state"], cs)
    np.testing.assert_array_equal(r["q_hat"], qh)
    np.testing.assert_array_equal(r["g"], g)


def test_layer_with_selection_projections_is_the_core():
    """Projections that select disjoint column blocks of h (hidden = CD + Hv*dv
    + 2 Hv) and an out_proj that puts y in the first Hv*dv columns: the layer is
    the core on those blocks, exactly (bf16-valued inputs are left unchanged by
    the bf16 rounding).  A transposed weight, or two projections fed to the
    wrong core inputs, fails it."""
    d = _dims(act="sigmoid")
    cd, vd, hv = d.conv_dim, d.n_v_heads * d.d_v, d.n_v_heads
    hidden = cd + vd + 2 * hv
    case = _rng_case(d, [9, 4], seed=73)
    rng = np.random.default_rng(74)
    h = oracle.round_bf16(rng.normal(size=(int(case["cu"][-1]), hidden)))
    eye = np.eye(hidden)
    w_qkv, w_z = eye[:cd], eye[cd:cd + vd]
    w_a, w_b = eye[cd + vd:cd + vd + hv], eye[cd + vd + hv:]
    w_out = np.zeros((hidden, vd))
    w_out[:vd] = np.eye(vd)
    r = oracle.layer(d, case["cu"], h, w_qkv, w_z, w_a, w_b, w_out, case["conv_w"],
                     case["A_log"], case["dt_bias"], case["norm_w"], case["conv_state"],
                     case["state"])
    x, z = h[:, :cd], h[:, cd:cd + vd]
    a, b = h[:, cd + vd:cd + vd + hv], h[:, cd + vd + hv:]
    ref = oracle.gdn(d, case["cu"], x, z, a, b, case["conv_w"], case["A_log"], case["dt_bias"],
                     case["norm_w"], case["conv_state"], case["state"])
    np.testing.assert_array_equal(r["h_out"][:, :vd], oracle.round_bf16(ref["out"]))
    np.testing.assert_array_equal(r["h_out"][:, vd:], 0.0)
    np.testing.assert_array_equal(r["state"], ref["state"])


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(75)
    v = rng.normal(size=4096) * np.exp(rng.uniform(-20, 20, 4096))
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(v), want)


def test_tiled_head_map_is_the_contiguous_one_with_value_heads_permuted():
    """Value head h reading key head h % Hk (tiled) is, bit for bit, the
    contiguous map (key head j // R) run on the same heads renumbered j = hk R + r
    for h = hk + Hk r: every per-value-head input (v channels and their conv
    weights and history, z, a, b, A_log, dt_bias, state) moved with its head."""
    d_t = oracle.Dims(2, 6, 8, 8, 4, "sigmoid", head_map="tiled")
    d_c = oracle.Dims(2, 6, 8, 8, 4, "sigmoid")
    hk_n, hv_n, dv = 2, 6, 8
    rr = hv_n // hk_n
    case = _rng_case(d_c, [11, 5], seed=76)
    perm = np.empty(hv_n, dtype=int)  # contiguous slot j holds tiled head perm[j]
    for hk in range(hk_n):
        for r in range(rr):
            perm[hk * rr + r] = hk + hk_n * r
    kd = 2 * hk_n * 8

    def per_head(u, axis, width):
        shp = list(u.shape)
        v = u.reshape(shp[:axis] + [hv_n, width] + shp[axis + 1:])
        return np.take(v, perm, axis=axis).reshape(shp)

    def move(c):
        m = dict(c)
        m["x"] = np.concatenate([c["x"][:, :kd], per_head(c["x"][:, kd:], 1, dv)], axis=1)
        m["conv_w"] = np.concatenate([c["conv_w"][:kd], per_head(c["conv_w"][kd:], 0, dv)])
        m["conv_state"] = np.concatenate([c["conv_state"][:, :kd],
                                          per_head(c["conv_state"][:, kd:], 1, dv)], axis=1)
        m["z"] = per_head(c["z"], 1, dv)
        m["a"], m["b"] = c["a"][:, perm], c["b"][:, perm]
        m["A_log"], m["dt_bias"] = c["A_log"][perm], c["dt_bias"][perm]
        m["state"] = c["state"][:, perm]
        return m

    def run(d, c):
        return oracle.gdn(d, c["cu"], c["x"], c["z"], c["a"], c["b"], c["conv_w"], c["A_log"],
                          c["dt_bias"], c["norm_w"], c["conv_state"], c["state"])
    rt, rc = run(d_t, case), run(d_c, move(case))
    np.testing.assert_array_equal(per_head(rt["out"], 1, dv), rc["out"])
    np.testing.assert_array_equal(rt["state"][:, perm], rc["state"])


def test_decay_coefficient_form_equals_A_log_form():
    """Giving the decay coefficient A = -exp(A_log) itself (the GGUF ssm_a)
    gives the same gates and outputs as giving A_log."""
    d = _dims()
    d_coef = oracle.Dims(d.n_k_heads, d.n_v_heads, d.d_k, d.d_v, d.conv_k, d.act, decay_form="coef")
    case = _rng_case(d, [7, 9], seed=77)
    coef = -np.exp(case["A_log"])
    g1, _ = oracle.gates(d, case["a"], case["b"], case["A_log"], case["dt_bias"])
    g2, _ = oracle.gates(d_coef, case["a"], case["b"], coef, case["dt_bias"])
    np.testing.assert_allclose(g2, g1, rtol=1e-14, atol=0)
    r1 = oracle.gdn(d, case["cu"], case["x"], case["z"], case["a"], case["b"], case["conv_w"],
                    case["A_log"], case["dt_bias"], case["norm_w"], case["conv_state"], case["state"])
    r2 = oracle.gdn(d_coef, case["cu"], case["x"], case["z"], case["a"], case["b"], case["conv_w"],
                    coef, case["dt_bias"], case["norm_w"], case["conv_state"], case["state"])
    np.testing.assert_allclose(r2["out"], r1["out"], rtol=1e-12, atol=1e-14)


def test_per_channel_decay_with_equal_channels_is_the_scalar_rule():
    """One decay per key channel, all channels of a value head given the same
    gate input and bias: exactly the one-decay-per-head rule."""
    d = _dims()
    d_pc = oracle.Dims(d.n_k_heads, d.n_v_heads, d.d_k, d.d_v, d.conv_k, d.act,
                       per_channel_decay=True)
    case = _rng_case(d, [8, 5], seed=78)
    a_pc = np.repeat(case["a"], d.d_k, axis=1)
    dtb_pc = np.repeat(case["dt_bias"], d.d_k)
    run = lambda dd, a, dtb: oracle.gdn(dd, case["cu"], case["x"], case["z"], a, case["b"],  # noqa: E731
                                         case["conv_w"], case["A_log"], dtb, case["norm_w"],
                                         case["conv_state"], case["state"])
    r1, r2 = run(d, case["a"], case["dt_bias"]), run(d_pc, a_pc, dtb_pc)
    np.testing.assert_array_equal(r2["out"], r1["out"])
    np.testing.assert_array_equal(r2["state"], r1["state"])


def test_per_channel_decay_without_writes_decays_each_state_row():
    """beta = 0: the state only decays, row i (key channel i) by exp(sum_t g[t, h, i]),
    and the readout is the decayed state read by q (closed form)."""
    d = oracle.Dims(1, 2, 8, 4, 4, "silu", per_channel_decay=True)
    rng = np.random.default_rng(79)
    t = 6
    q = rng.normal(size=(t, 1, 8))
    k = rng.normal(size=(t, 1, 8))
    v = rng.normal(size=(t, 2, 4))
    g = -rng.uniform(0, 1, size=(t, 2, 8))
    s0 = rng.normal(size=(1, 2, 8, 4))
    o, s1, _ = oracle.recurrence(d, [0, t], q, k, v, g, np.zeros((t, 2)), s0)
    cum = np.cumsum(g, axis=0)  # [t, h, i]
    want_s = s0[0] * np.exp(cum[-1])[:, :, None]
    np.testing.assert_allclose(s1[0], want_s, rtol=1e-13, atol=1e-15)
    for tt in range(t):
        st = s0[0] * np.exp(cum[tt])[:, :, None]  # [h, i, dv]
        want_o = np.einsum("hij,i->hj", st, q[tt, 0])
        np.testing.assert_allclose(o[tt], want_o, rtol=1e-12, atol=1e-14)


def test_decode_steps_equal_one_prefill():
    """T one-token calls carrying (state, conv state) == one T-token call, and the
    per-token intermediate states equal the states after each single step."""
    d = _dims(act="sigmoid")
    case = _rng_case(d, [6], seed=81)
    args = (case["conv_w"], case["A_log"], case["dt_bias"], case["norm_w"])
    full = oracle.gdn(d, [0, 6], case["x"], case["z"], case["a"], case["b"], *args,
                      case["conv_state"], case["state"], want_inter=True)
    cs, s = case["conv_state"], case["state"]
    for i in range(6):
        r = oracle.gdn(d, [0, 1], case["x"][i:i + 1], case["z"][i:i + 1], case["a"][i:i + 1],
                       case["b"][i:i + 1], *args, cs, s)
        np.testing.assert_allclose(r["out"][0], full["out"][i], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r["state"][0], full["inter"][i], rtol=1e-12, atol=1e-14)
        cs, s = r["conv_state"], r["state"]
    np.testing.assert_allclose(s, full["state"], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(cs, full["conv_state"])


def test_workload_generator_shapes_and_bf16_rounding():
    c = workloads.config(0)
    assert c.x.shape == (64, 256) and c.conv_w.shape == (256, 4) and c.x.dtype == np.float32
    assert c.state is None and c.conv_state is None
    c4 = workloads.generate("t", n_k_heads=2, n_v_heads=4, d_k=8, d_v=8, mode="decode", n_seq=3,
                            tokens_per_seq=4, dtype="bf16", state_std=0.05, conv_state_std=1.0)
    bits = c4.x.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)        # bf16-representable
    assert c4.cu_seqlens.tolist() == [0, 4, 8, 12]
    np.testing.assert_array_equal(workloads.round_bf16(np.array([1.0 + 2 ** -8], np.float32)), [1.0])
    np.testing.assert_array_equal(workloads.round_bf16(np.array([1.0 + 3 * 2 ** -8], np.float32)),
                                  [1.0 + 2 ** -6])
    ref = torch.tensor(c4.z.ravel()[:100] + np.float32(1e-3)).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(workloads.round_bf16(c4.z.ravel()[:100] + np.float32(1e-3)), ref)


def test_bf16_half_ulp_helper():
    """The test metric's storage-rounding allowance: exact half ulps of bf16 values."""
    from gdn_cases import bf16_half_ulp
    v = np.array([1.0, 1.5, -2.0, 3.0, 0.0, 2.0 ** -10])
    np.testing.assert_array_equal(bf16_half_ulp(v), [2 ** -8, 2 ** -8, 2 ** -7, 2 ** -7, 0.0, 2 ** -18])
    # any float32 rounds to bf16 within half an ulp of the result
    x = np.random.default_rng(0).normal(size=1000).astype(np.float32) * 37
    r = workloads.round_bf16(x).astype(np.float64)
    assert np.all(np.abs(r - x) <= bf16_half_ulp(r) * (1 + 1e-12))
