/*
 * Gated DeltaNet mixer core -- CPU oracle in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header or constant with the CUDA library, and nothing on the product path
 * may link it: only the tests, the smoke check and the benchmark's CPU
 * baseline leg load it.
 *
 * Every step is written in the order and notation of the pages that define
 * it:
 *   [cpu.rs]  cherenkov qwen4_exp/cpu.rs -- `deltanet` (decode form) and
 *             `causal_conv`
 *   [qwen.rs] oxinfer 0.0.5 src/qwen.rs -- `gdn_forward` (prefill over t
 *             tokens), `DeltaRule::run`, `GdnState`
 * Readings taken where the pages are silent or disagree are noted at each
 * function (output-gate activation is a parameter; conv state is
 * [seq][channel][K-1], oldest first; eps values are parameters).
 *
 * Layouts (all row-major, token-major packed like [qwen.rs] gdn_forward):
 *   x       [T_total, CD]        CD = 2*Hk*dk + Hv*dv, channels [q | k | v]
 *   z       [T_total, Hv*dv]
 *   a, b    [T_total, Hv]
 *   conv_w  [CD, K]              tap K-1 multiplies the current token
 *   conv_state [n_seq, CD, K-1]  oldest first
 *   state   [n_seq, Hv, dk, dv]  key lane major ("[key_lane][value_lane]")
 *   inter   [T_total, Hv, dk, dv] state after every token (optional)
 *   out     [T_total, Hv*dv]
 * Sequences are delimited by cu_seqlens[n_seq+1] (packed, like varlen
 * prefill); each sequence has its own conv history and recurrent state.
 *
 * parity: every function here is pinned by tests/test_oracle_pins.py.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <tgmath.h>

/* The arithmetic type.  The parity build is double (the default); the CPU
 * baseline that the benchmark times is the same code built with
 * -DORACLE_REAL=float (tgmath.h picks exp/sqrt/log1p of that type).  The eps
 * fields of oracle_dims stay double in both builds. */
#ifndef ORACLE_REAL
#define ORACLE_REAL double
#endif
typedef ORACLE_REAL real;

typedef struct {
    int32_t n_k_heads;  /* Hk: linear_num_key_heads   */
    int32_t n_v_heads;  /* Hv: linear_num_value_heads */
    int32_t d_k;        /* linear_key_head_dim        */
    int32_t d_v;        /* linear_value_head_dim      */
    int32_t conv_k;     /* linear_conv_kernel_dim (K) */
    int32_t act;        /* output gate: 0 = SiLU, 1 = sigmoid */
    double l2_eps;      /* 1e-6 on both pages */
    double rms_eps;     /* 1e-6 on cpu.rs; rms_norm_eps on qwen.rs */
    int32_t tiled;      /* key head of value head hv: hv % Hk if 1, hv / (Hv/Hk) if 0 */
    int32_t decay_coef; /* A_log[] holds the decay coefficient itself if 1 */
    int32_t per_channel; /* 1: a decay per key channel (a [T,Hv,dk], dt_bias [Hv,dk]) */
} oracle_dims;

static int conv_dim(const oracle_dims* d) {
    return 2 * d->n_k_heads * d->d_k + d->n_v_heads * d->d_v;
}

static real sigmoid(real x) { return 1.0 / (1.0 + exp(-x)); }
static real silu(real x) { return x * sigmoid(x); }

/* [qwen.rs] DeltaRule::run: softplus is the identity above 20, else
 * ln(1 + e^x).  log1p is the same function with less rounding. */
static real softplus(real x) { return x > 20.0 ? x : log1p(exp(x)); }

/*
 * Step a1 + a2: causal depthwise conv with SiLU, and the conv-state update.
 * [qwen.rs] gdn_forward, "Causal depthwise conv over time": output i of a
 * sequence is sum_j w[ch,j] * src(i-(K-1)+j, ch), where a negative source
 * index reads the conv history (slot K-1+i), then s*sigmoid(s).
 * [qwen.rs] gdn_forward, "Update conv state with the last kc-1 raw inputs":
 * slot s of the new history holds raw input t-(K-1)+s, or the old history
 * when the sequence is shorter than K-1.  [cpu.rs] causal_conv is the t=1
 * case of both.
 * conv_state_in == NULL means an all-zero history; conv_state_out may be
 * NULL, and may alias conv_state_in.
 */
void oracle_conv(const oracle_dims* d, int n_seq, const int32_t* cu_seqlens,
                 const real* x, const real* conv_w,
                 const real* conv_state_in, real* c, real* conv_state_out) {
    const int cd = conv_dim(d);
    const int kc = d->conv_k;
    const int keep = kc - 1;
    for (int n = 0; n < n_seq; ++n) {
        const int bos = cu_seqlens[n];
        const int len = cu_seqlens[n + 1] - bos;
#pragma omp parallel for schedule(static)
        for (int i = 0; i < len; ++i) {
            for (int ch = 0; ch < cd; ++ch) {
                real s = 0.0;
                for (int j = 0; j < kc; ++j) {
                    const int src = i - (kc - 1) + j;
                    real v;
                    if (src >= 0) {
                        v = x[(size_t)(bos + src) * cd + ch];
                    } else if (conv_state_in) {
                        v = conv_state_in[((size_t)n * cd + ch) * keep + (keep + src)];
                    } else {
                        v = 0.0;
                    }
                    s += conv_w[(size_t)ch * kc + j] * v;
                }
                c[(size_t)(bos + i) * cd + ch] = silu(s);
            }
        }
    }
    if (!conv_state_out || keep == 0) return;
    for (int n = 0; n < n_seq; ++n) {
        const int bos = cu_seqlens[n];
        const int len = cu_seqlens[n + 1] - bos;
        for (int ch = 0; ch < cd; ++ch) {
            real nw[8];
            for (int slot = 0; slot < keep; ++slot) {
                const int ti = len - keep + slot;
                if (ti >= 0) {
                    nw[slot] = x[(size_t)(bos + ti) * cd + ch];
                } else if (conv_state_in) {
                    nw[slot] = conv_state_in[((size_t)n * cd + ch) * keep + (keep + ti)];
                } else {
                    nw[slot] = 0.0;
                }
            }
            for (int slot = 0; slot < keep; ++slot)
                conv_state_out[((size_t)n * cd + ch) * keep + slot] = nw[slot];
        }
    }
}

/*
 * Step a3: per token and key head, q and k are L2-normalised over d_k as
 * x * (sum x^2 + eps)^(-1/2); only q is then scaled by d_k^(-1/2).
 * [qwen.rs] DeltaRule::run (qn_inv, kn_inv, qscale); [cpu.rs] deltanet,
 * "only q receives 1/sqrt(dk)".  v is passed through unchanged.
 * Outputs: q_hat, k_hat [T, Hk, dk]; v [T, Hv, dv].
 */
void oracle_normalize(const oracle_dims* d, int n_tok, const real* c,
                      real* q_hat, real* k_hat, real* v) {
    const int cd = conv_dim(d);
    const int hk_n = d->n_k_heads, dk = d->d_k;
    const int key_dim = hk_n * dk, value_dim = d->n_v_heads * d->d_v;
    const real qscale = 1.0 / sqrt((real)dk);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < n_tok; ++t) {
        const real* row = c + (size_t)t * cd;
        for (int h = 0; h < hk_n; ++h) {
            const real* qv = row + h * dk;
            const real* kv = row + key_dim + h * dk;
            real qss = 0.0, kss = 0.0;
            for (int i = 0; i < dk; ++i) {
                qss += qv[i] * qv[i];
                kss += kv[i] * kv[i];
            }
            const real qn_inv = 1.0 / sqrt(qss + d->l2_eps);
            const real kn_inv = 1.0 / sqrt(kss + d->l2_eps);
            for (int i = 0; i < dk; ++i) {
                q_hat[((size_t)t * hk_n + h) * dk + i] = qv[i] * qn_inv * qscale;
                k_hat[((size_t)t * hk_n + h) * dk + i] = kv[i] * kn_inv;
            }
        }
        memcpy(v + (size_t)t * value_dim, row + 2 * key_dim, sizeof(real) * value_dim);
    }
}

/*
 * Step a4: write strength beta = sigmoid(b) and log-decay
 * g = decay_coef * softplus(a + dt_bias), per token and value head.
 * [qwen.rs] DeltaRule::run (beta, ga, softplus, decay) with the loader's
 * decay_coef = -exp(A_log), or the GGUF ssm_a read as decay_coef directly
 * (d->decay_coef); [cpu.rs] deltanet (beta, g, decay = g.exp()).
 */
void oracle_gates(const oracle_dims* d, int n_tok, const real* a, const real* b,
                  const real* A_log, const real* dt_bias, real* g, real* beta) {
    const int hv_n = d->n_v_heads;
    const int nc = d->per_channel ? d->d_k : 1; /* decays per value head */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < n_tok; ++t) {
        for (int h = 0; h < hv_n; ++h) {
            const size_t i = (size_t)t * hv_n + h;
            beta[i] = sigmoid(b[i]);
            const real coef = d->decay_coef ? A_log[h] : -exp(A_log[h]);
            for (int j = 0; j < nc; ++j)
                g[i * nc + j] = coef * softplus(a[i * nc + j] + dt_bias[(size_t)h * nc + j]);
        }
    }
}

/*
 * Step a5: the gated delta rule in its recurrent form, token by token.
 * [cpu.rs] deltanet and [qwen.rs] DeltaRule::run, per value head hv with key
 * head hk = hv / (Hv/Hk) (contiguous groups), or hk = hv % Hk when d->tiled
 * (qwen.rs DeltaRule::run's `tiled`):
 *   S <- exp(g) * S                (decay first)
 *   kv = S^T k                     (read of the decayed state)
 *   delta = beta * (v - kv)
 *   S <- S + k delta^T             (rank-one write)
 *   o = S^T q                      (readout of the written state)
 * The loops keep the pages' order: rows ik outer, value lanes iv inner.
 * state_in == NULL means S = 0; state_out may alias state_in or be NULL.
 * inter (optional) receives the state after every token, [T, Hv, dk, dv].
 * o is [T, Hv, dv].  Value heads are independent (the pages run them on a
 * thread pool); this loop runs them on OpenMP threads in the same way.
 */
void oracle_recurrence(const oracle_dims* d, int n_seq, const int32_t* cu_seqlens,
                       const real* q_hat, const real* k_hat, const real* v,
                       const real* g, const real* beta,
                       const real* state_in, real* state_out, real* inter, real* o) {
    const int hk_n = d->n_k_heads, hv_n = d->n_v_heads, dk = d->d_k, dv = d->d_v;
    const int group = hv_n / hk_n;
    const size_t slab = (size_t)dk * dv;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int n = 0; n < n_seq; ++n) {
        for (int hv = 0; hv < hv_n; ++hv) {
            const int hk = d->tiled ? hv % hk_n : hv / group;
            const int bos = cu_seqlens[n];
            const int len = cu_seqlens[n + 1] - bos;
            real* s = (real*)malloc(sizeof(real) * slab);
            real* kv_mem = (real*)malloc(sizeof(real) * dv);
            real* delta = (real*)malloc(sizeof(real) * dv);
            if (state_in)
                memcpy(s, state_in + ((size_t)n * hv_n + hv) * slab, sizeof(real) * slab);
            else
                memset(s, 0, sizeof(real) * slab);
            for (int i = 0; i < len; ++i) {
                const size_t t = (size_t)bos + i;
                const real* qh = q_hat + (t * hk_n + hk) * dk;
                const real* kh = k_hat + (t * hk_n + hk) * dk;
                const real* vh = v + (t * hv_n + hv) * dv;
                /* one decay per value head, or one per key channel (row ik) */
                const real* gt = g + (t * hv_n + hv) * (d->per_channel ? dk : 1);
                const real bt = beta[t * hv_n + hv];
                for (int iv = 0; iv < dv; ++iv) kv_mem[iv] = 0.0;
                for (int ik = 0; ik < dk; ++ik) {
                    real* row = s + (size_t)ik * dv;
                    const real decay = exp(gt[d->per_channel ? ik : 0]);
                    for (int iv = 0; iv < dv; ++iv) {
                        row[iv] *= decay;
                        kv_mem[iv] += row[iv] * kh[ik];
                    }
                }
                for (int iv = 0; iv < dv; ++iv) delta[iv] = (vh[iv] - kv_mem[iv]) * bt;
                real* oh = o + (t * hv_n + hv) * dv;
                for (int iv = 0; iv < dv; ++iv) oh[iv] = 0.0;
                for (int ik = 0; ik < dk; ++ik) {
                    real* row = s + (size_t)ik * dv;
                    for (int iv = 0; iv < dv; ++iv) {
                        row[iv] += kh[ik] * delta[iv];
                        oh[iv] += row[iv] * qh[ik];
                    }
                }
                if (inter) memcpy(inter + (t * hv_n + hv) * slab, s, sizeof(real) * slab);
            }
            if (state_out)
                memcpy(state_out + ((size_t)n * hv_n + hv) * slab, s, sizeof(real) * slab);
            free(s);
            free(kv_mem);
            free(delta);
        }
    }
}

/*
 * Step a6: gated RMSNorm per token and value head over d_v:
 * y = o * (mean(o^2) + eps)^(-1/2) * norm_w * act(z), with a plain weight
 * (no 1 + w) shared by all heads.  [qwen.rs] gdn_forward, "Gated RMSNorm per
 * head" (SiLU gate); [cpu.rs] deltanet (rms_norm then sigmoid gate when
 * output_gate_type is "sigmoid").  act: 0 = SiLU, 1 = sigmoid.
 */
void oracle_gated_norm(const oracle_dims* d, int n_tok, const real* o, const real* z,
                       const real* norm_w, real* y) {
    const int hv_n = d->n_v_heads, dv = d->d_v;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < n_tok; ++t) {
        for (int h = 0; h < hv_n; ++h) {
            const size_t base = ((size_t)t * hv_n + h) * dv;
            real ss = 0.0;
            for (int j = 0; j < dv; ++j) ss += o[base + j] * o[base + j];
            const real r = 1.0 / sqrt(ss / dv + d->rms_eps);
            for (int j = 0; j < dv; ++j) {
                const real zz = z[base + j];
                const real gate = d->act == 1 ? sigmoid(zz) : silu(zz);
                y[base + j] = o[base + j] * r * norm_w[j] * gate;
            }
        }
    }
}

/*
 * The whole mixer core, a1..a6 in order, as [qwen.rs] gdn_forward runs it
 * between the input projections and out_proj.  Scratch is allocated here.
 * Optional outputs (NULL to skip): conv_state_out, state_out, inter, and the
 * stage outputs q_hat/k_hat [T,Hk,dk], v_out [T,Hv,dv], g_out/beta_out [T,Hv].
 * Returns 0, or -1 when scratch could not be allocated.
 */
int oracle_gdn(const oracle_dims* d, int n_seq, const int32_t* cu_seqlens,
               const real* x, const real* z, const real* a, const real* b,
               const real* conv_w, const real* A_log, const real* dt_bias,
               const real* norm_w,
               const real* conv_state_in, real* conv_state_out,
               const real* state_in, real* state_out, real* inter, real* out,
               real* q_hat_out, real* k_hat_out, real* v_out,
               real* g_out, real* beta_out) {
    const int cd = conv_dim(d);
    const size_t n_tok = (size_t)cu_seqlens[n_seq];
    const size_t key_n = n_tok * d->n_k_heads * d->d_k;
    const size_t val_n = n_tok * d->n_v_heads * d->d_v;
    const size_t gate_n = n_tok * d->n_v_heads;
    const size_t decay_n = gate_n * (d->per_channel ? d->d_k : 1);
    real* c = (real*)malloc(sizeof(real) * (n_tok * cd + 1));
    real* qh = q_hat_out ? q_hat_out : (real*)malloc(sizeof(real) * (key_n + 1));
    real* kh = k_hat_out ? k_hat_out : (real*)malloc(sizeof(real) * (key_n + 1));
    real* vv = v_out ? v_out : (real*)malloc(sizeof(real) * (val_n + 1));
    real* gg = g_out ? g_out : (real*)malloc(sizeof(real) * (decay_n + 1));
    real* bb = beta_out ? beta_out : (real*)malloc(sizeof(real) * (gate_n + 1));
    real* o = (real*)malloc(sizeof(real) * (val_n + 1));
    int rc = 0;
    if (!c || !qh || !kh || !vv || !gg || !bb || !o) {
        rc = -1;
    } else {
        oracle_conv(d, n_seq, cu_seqlens, x, conv_w, conv_state_in, c, conv_state_out);
        oracle_normalize(d, (int)n_tok, c, qh, kh, vv);
        oracle_gates(d, (int)n_tok, a, b, A_log, dt_bias, gg, bb);
        oracle_recurrence(d, n_seq, cu_seqlens, qh, kh, vv, gg, bb, state_in, state_out, inter, o);
        oracle_gated_norm(d, (int)n_tok, o, z, norm_w, out);
    }
    free(c);
    if (!q_hat_out) free(qh);
    if (!k_hat_out) free(kh);
    if (!v_out) free(vv);
    if (!g_out) free(gg);
    if (!beta_out) free(bb);
    free(o);
    return rc;
}
