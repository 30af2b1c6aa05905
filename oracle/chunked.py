"""Second, independent formulation of the delta rule: the chunked (WY / UT) form.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  This file exists to pin
the token-by-token recurrence in ``gdn_oracle.c``: the two are written from
different derivations and agree only if both are right.

Derivation, from the recurrence of the pages ([cpu.rs] ``deltanet``, [qwen.rs]
``DeltaRule::run``): S_t = e^{g_t} S_{t-1} + k_t u_t^T with
u_t = beta_t (v_t - (e^{g_t} S_{t-1})^T k_t).  Within a chunk that starts from
state S0, let G_t = sum_{s<=t} g_s.  Unrolling gives
    S_t = e^{G_t} S0 + sum_{s<=t} e^{G_t-G_s} k_s u_s^T,
so the u_t solve the unit-lower-triangular system (I + A) U = diag(beta) V -
diag(beta e^G) K S0 with A_ts = beta_t e^{G_t-G_s} k_t.k_s for s < t.  Hence,
with T = (I + A)^{-1}:
    W = T diag(beta e^G) K,   U~ = T diag(beta) V,   U = U~ - W S0
    O = diag(e^G) Q S0 + (M o Q K^T) U,   M_ts = e^{G_t-G_s} for s <= t, else 0
    S_end = e^{G_last} S0 + K^T diag(e^{G_last - G}) U
With one decay per key channel (g_t a vector) the same steps hold with diag(e^{g_t})
for e^{g_t}; ``chunk_step_per_channel`` forms the pairwise factors per channel.
All arithmetic is float64 numpy; nothing is shared with the C oracle.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg


def chunk_step(q, k, v, g, beta, s0):
    """One chunk for one value head.

    q, k: [C, dk]; v: [C, dv]; g, beta: [C]; s0: [dk, dv].
    Returns (o [C, dv], s_end [dk, dv]).
    """
    c = q.shape[0]
    G = np.cumsum(g)
    diff = G[:, None] - G[None, :]
    lower = np.tril(np.ones((c, c), dtype=bool), k=-1)
    A = np.where(lower, beta[:, None] * np.exp(np.where(lower, diff, 0.0)) * (k @ k.T), 0.0)
    eye = np.eye(c)
    # T = (I + A)^{-1} applied by a unit-lower-triangular solve.
    rhs_w = (beta * np.exp(G))[:, None] * k
    rhs_u = beta[:, None] * v
    W = scipy.linalg.solve_triangular(eye + A, rhs_w, lower=True, unit_diagonal=True)
    U_t = scipy.linalg.solve_triangular(eye + A, rhs_u, lower=True, unit_diagonal=True)
    U = U_t - W @ s0
    causal = np.tril(np.ones((c, c), dtype=bool))
    M = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
    o = np.exp(G)[:, None] * (q @ s0) + (M * (q @ k.T)) @ U
    s_end = np.exp(G[-1]) * s0 + k.T @ (np.exp(G[-1] - G)[:, None] * U)
    return o, s_end


def chunk_step_per_channel(q, k, v, g, beta, s0):
    """One chunk for one value head with one decay per key channel.

    q, k: [C, dk]; v: [C, dv]; g: [C, dk]; beta: [C]; s0: [dk, dv].
    Returns (o [C, dv], s_end [dk, dv]).

    The same unrolling with diag(e^{g_t}) in place of e^{g_t}: with
    G_t = sum_{s<=t} g_s (a vector over the key channels),
        S_t = diag(e^{G_t}) S0 + sum_{s<=t} diag(e^{G_t-G_s}) k_s u_s^T,
    so A_ts = beta_t sum_i k_t,i k_s,i e^{G_t,i-G_s,i} (s < t) and
        W = T diag(beta) (K o e^G),   U~ = T diag(beta) V,   U = U~ - W S0
        O = (Q o e^G) S0 + M U,   M_ts = sum_i q_t,i k_s,i e^{G_t,i-G_s,i} (s <= t)
        S_end = diag(e^{G_last}) S0 + (K o e^{G_last-G})^T U.
    The pairwise factors are formed per (t, s, i) from differences of G, only
    where s <= t (each then at most 1).
    """
    c = q.shape[0]
    G = np.cumsum(g, axis=0)                                   # [C, dk]
    lower = np.tril(np.ones((c, c), dtype=bool), k=-1)
    causal = np.tril(np.ones((c, c), dtype=bool))
    diff = G[:, None, :] - G[None, :, :]                       # [t, s, i]
    E = np.exp(np.where(causal[:, :, None], diff, 0.0))
    A = np.where(lower, beta[:, None] * np.einsum("ti,si,tsi->ts", k, k, E), 0.0)
    M = np.where(causal, np.einsum("ti,si,tsi->ts", q, k, E), 0.0)
    eye = np.eye(c)
    W = scipy.linalg.solve_triangular(eye + A, beta[:, None] * (k * np.exp(G)), lower=True,
                                      unit_diagonal=True)
    U_t = scipy.linalg.solve_triangular(eye + A, beta[:, None] * v, lower=True, unit_diagonal=True)
    U = U_t - W @ s0
    o = (q * np.exp(G)) @ s0 + M @ U
    s_end = np.exp(G[-1])[:, None] * s0 + (k * np.exp(G[-1] - G)).T @ U
    return o, s_end


def recurrence_chunked(cu_seqlens, q_hat, k_hat, v, g, beta, state=None, chunk=16,
                       v_to_k=None):
    """The delta rule over packed sequences in chunks of ``chunk`` tokens.

    q_hat, k_hat: [T, Hk, dk]; v: [T, Hv, dv]; g: [T, Hv] (or [T, Hv, dk], one
    decay per key channel); beta: [T, Hv];
    state: [N, Hv, dk, dv] or None (zeros).  Value head h reads key head
    ``v_to_k(h)``; by default contiguous groups h // (Hv // Hk).
    Returns (o [T, Hv, dv], final state [N, Hv, dk, dv]).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = cu.size - 1
    t_total, hk_n, dk = q_hat.shape
    hv_n, dv = v.shape[1], v.shape[2]
    if v_to_k is None:
        grp = hv_n // hk_n
        v_to_k = lambda h: h // grp  # noqa: E731
    o = np.zeros((t_total, hv_n, dv))
    s_out = np.zeros((n, hv_n, dk, dv))
    for i in range(n):
        bos, eos = int(cu[i]), int(cu[i + 1])
        for h in range(hv_n):
            hk = v_to_k(h)
            s = np.zeros((dk, dv)) if state is None else np.array(state[i, h], dtype=np.float64)
            for c0 in range(bos, eos, chunk):
                c1 = min(c0 + chunk, eos)
                step = chunk_step_per_channel if g.ndim == 3 else chunk_step
                oc, s = step(q_hat[c0:c1, hk], k_hat[c0:c1, hk], v[c0:c1, h],
                             g[c0:c1, h], beta[c0:c1, h], s)
                o[c0:c1, h] = oc
            s_out[i, h] = s
    return o, s_out
