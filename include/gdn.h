/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) mixer core for GB300 (sm_103a).
 *
 * The core is what runs between a GDN layer's input projections and its
 * out_proj (oxinfer 0.0.5 src/qwen.rs, fn gdn_forward; cherenkov
 * qwen4_exp/cpu.rs, fn deltanet):
 *   a1  causal depthwise conv over the packed [q | k | v] channels, then SiLU
 *   a2  conv-state update: the last K-1 raw inputs of each sequence
 *   a3  per key head, q and k L2-normalised over d_k; q scaled by d_k^-1/2
 *   a4  beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias)
 *   a5  per value head, token by token: S <- exp(g) S; u = beta (v - S^T k);
 *       S <- S + k u^T; o = S^T q    (qwen.rs DeltaRule::run, cpu.rs deltanet)
 *   a6  y = norm_w * o * (mean(o^2) + eps)^-1/2 * act(z), act = SiLU or sigmoid
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer is a DEVICE pointer unless its name ends in _host.  The
 *   caller allocates and owns every buffer; no call allocates device memory
 *   or keeps a pointer after it returns.
 * - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *   is the legacy default stream).  Returning GDN_OK means the work was
 *   validated and enqueued, not that it has finished.
 * - Layouts are row-major and token-major ("packed"): sequence i owns tokens
 *   [cu_seqlens[i], cu_seqlens[i+1]) of every [T, ...] array.
 *     x       [T, CD]   CD = 2*Hk*dk + Hv*dv, channels [q | k | v]
 *     z       [T, Hv*dv]
 *     a, b    [T, Hv]
 *     out     [T, Hv*dv]
 *     state   [N, Hv, dk, dv]  fp32, key lane major (row = key lane)
 *     conv_state [N, CD, K-1]  activation dtype, oldest input first
 *   Activations (x, z, a, b, out, conv_state, qkv_out) are all fp32 or all
 *   bf16 (gdn_dims.dtype).  Parameters and recurrent states are always fp32.
 * - Value head h reads key head h / (Hv/Hk) (contiguous groups).
 * - Errors: each call returns a gdn_status; on failure nothing was enqueued
 *   (or, for GDN_ERR_CUDA, a launch failed), and gdn_last_error() returns a
 *   message naming the call and the reason.  No call aborts the process.
 * - Buffers must be 16-byte aligned (x, z, out, states, qkv_out; with
 *   per-channel decay, a as well in gdn_prefill).
 * - A call takes at most GDN_MAX_SEQUENCES sequences (kernels index them on
 *   the second grid dimension); larger batches are refused before any launch.
 * - Failure injection (testing a caller's failure path, as cortiq-engine
 *   0.8.76 pipeline.rs does with its test-only nll_test_fail_at): the environment variable GDN_FAULT
 *   is a comma-separated list of sites -- conv, prefill, decode, verify,
 *   commit, layer, or all.  A call whose site is listed validates its
 *   arguments, then returns GDN_ERR_INJECTED without enqueuing anything, so
 *   every caller buffer is left as it was.  The site stall_scan is a device
 *   test hook: a bf16 prefill that takes the fused tensor-core launch makes
 *   its scan wait (for at most 1 ms) on a chunk flag that nothing sets, so
 *   that the bounded wait runs out; the call returns GDN_OK and the next
 *   gdn_sync_status reports GDN_ERR_TIMEOUT.  GDN_FAULT is read on every call.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

/* Most sequences one call takes (the CUDA grid's second dimension). */
#define GDN_MAX_SEQUENCES 65535

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null pointer, bad size or cu_seqlens, misalignment */
    GDN_ERR_UNSUPPORTED = 2, /* geometry the kernels are not built for */
    GDN_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    GDN_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
    GDN_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (gdn_sync_status) */
    GDN_ERR_INJECTED = 6     /* a fault injected through GDN_FAULT (testing) */
} gdn_status;

typedef enum gdn_dtype { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 } gdn_dtype;

/* Output-gate activation: qwen.rs gdn_forward uses SiLU, cpu.rs deltanet and
 * the qwen4_exp config (output_gate_sigmoid) use sigmoid. */
typedef enum gdn_act { GDN_ACT_SILU = 0, GDN_ACT_SIGMOID = 1 } gdn_act;

/* Which key head a value head reads (qwen.rs DeltaRule::run): h / (Hv/Hk),
 * contiguous groups (cpu.rs deltanet, the safetensors checkpoints), or h % Hk,
 * tiled (the GGUF checkpoints' layout). */
typedef enum gdn_head_map { GDN_HEADS_CONTIGUOUS = 0, GDN_HEADS_TILED = 1 } gdn_head_map;

/* What gdn_params.A_log holds (qwen.rs loader, decay_coef): log A, the
 * checkpoint's A_log, so that g = -exp(A_log) softplus(a + dt_bias); or the
 * decay coefficient itself (GGUF ssm_a, which stores -exp(A_log)), so that
 * g = A_log[h] softplus(a + dt_bias). */
typedef enum gdn_decay_form { GDN_DECAY_A_LOG = 0, GDN_DECAY_COEF = 1 } gdn_decay_form;

/* Geometry (names of qwen4_exp.rs GdnCfg / qwen.rs QwenConfig).
 * Supported: d_k, d_v in {32, 64, 128}; 2 <= conv_k <= 4;
 * n_v_heads a multiple of n_k_heads; eps > 0. */
typedef struct gdn_dims {
    int32_t n_k_heads; /* Hk  linear_num_key_heads */
    int32_t n_v_heads; /* Hv  linear_num_value_heads */
    int32_t d_k;       /* linear_key_head_dim */
    int32_t d_v;       /* linear_value_head_dim */
    int32_t conv_k;    /* K   linear_conv_kernel_dim */
    int32_t dtype;     /* gdn_dtype of the activations */
    int32_t act;       /* gdn_act of the output gate */
    float l2_eps;      /* q/k L2-norm eps (1e-6 on the pages) */
    float rms_eps;     /* gated RMSNorm eps (1e-6 / rms_norm_eps) */
    int32_t head_map;  /* gdn_head_map; 0 (contiguous) when zero-initialised */
    int32_t decay_form; /* gdn_decay_form; 0 (A_log) when zero-initialised */
    /* 1: one decay per key channel (the per-channel decayed delta rule of the
     * pages' Kimi Delta Attention mixer, qwen.rs Mixer::Kda): S <- diag(e^g) S
     * with g [T, Hv, dk] = coef[h] softplus(a[t, h, i] + dt_bias[h, i]); the
     * gate input a is then [T, Hv*dk] and dt_bias [Hv*dk] (b stays [T, Hv]).
     * A bf16 prefill with d_k = d_v = 128 runs it on the chunked tensor-core
     * path, everything else on the token-recurrent kernel;
     * gdn_layer_prefill refuses it.
     * 0 (one decay per value head) when zero-initialised. */
    int32_t decay_per_channel;
} gdn_dims;

/* Per-layer parameters, fp32 device pointers (qwen.rs loader: conv1d.weight
 * [CD,1,K], A_log [Hv], dt_bias [Hv], norm.weight [dv], plain weight). */
typedef struct gdn_params {
    const float* conv_w;  /* [CD, K]; tap K-1 multiplies the current token */
    const float* A_log;   /* [Hv] */
    const float* dt_bias; /* [Hv] */
    const float* norm_w;  /* [dv] */
} gdn_params;

/*
 * gdn_conv -- steps a1..a4 only (the prologue), for callers that run their
 * own recurrence, and for tests.
 *   x [T, CD]; a, b [T, Hv]; cu_seqlens [n_seq+1] (device) and the same values
 *   on the host (cu_seqlens_host), which is validated and used for sizing.
 *   conv_state_in [N, CD, K-1] or NULL (all-zero history).
 *   conv_state_out [N, CD, K-1] or NULL (not written); may equal conv_state_in.
 *   qkv_out [T, CD]: [q_hat (already scaled by d_k^-1/2) | k_hat | v], in the
 *   activation dtype.  g_out, beta_out [T, Hv] fp32 (g is the log-decay).
 * Defined by qwen.rs gdn_forward (conv, conv-state update) and
 * DeltaRule::run (normalisation, gates).
 */
gdn_status gdn_conv(const gdn_dims* dims, const gdn_params* params, int32_t n_seq,
                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                    const void* x, const void* a, const void* b,
                    const void* conv_state_in, void* conv_state_out,
                    void* qkv_out, float* g_out, float* beta_out, void* stream);

/*
 * gdn_prefill_workspace_size -- bytes of device workspace gdn_prefill needs
 * for this geometry and sequence layout (written to *bytes; may be 0).
 */
gdn_status gdn_prefill_workspace_size(const gdn_dims* dims, int32_t n_seq,
                                      const int32_t* cu_seqlens_host, size_t* bytes);

/*
 * gdn_prefill -- the whole core (a1..a6) over n_seq packed sequences of any
 * lengths (qwen.rs gdn_forward over t tokens; each sequence independent, with
 * its own conv history and recurrent state).
 *   initial_state [N, Hv, dk, dv] or NULL (zeros).  final_state: same shape,
 *   or NULL (not written); may equal initial_state.
 *   conv_state_in / conv_state_out as in gdn_conv (NULL allowed).
 *   out [T, Hv*dv] in the activation dtype.
 *   workspace: at least gdn_prefill_workspace_size() bytes, 256-byte aligned.
 * bf16 activations run the chunked form on tensor cores (bf16 operands, fp32
 * accumulation and fp32 state), with scalar or per-channel decay; fp32
 * activations run the token recurrence in fp32 on CUDA cores.
 */
gdn_status gdn_prefill(const gdn_dims* dims, const gdn_params* params, int32_t n_seq,
                       const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                       const void* x, const void* z, const void* a, const void* b,
                       const void* conv_state_in, void* conv_state_out,
                       const float* initial_state, float* final_state, void* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_prefill_noalloc -- gdn_prefill for callers that cannot allocate device
 * memory: an engine plugin that is given its inputs and outputs but no
 * workspace, or a serving loop whose memory is fixed before the first request
 * and that may not call cudaMalloc (or a framework allocator) on its path.
 * The pages have no counterpart: their CPU loop needs no scratch memory.
 *   Arguments are those of gdn_prefill without the workspace; the scratch is
 *   a built-in device array of gdn_prefill_noalloc_scratch_bytes() bytes
 *   (64 MiB).  It becomes resident on a device when the library's module is
 *   loaded there -- under CUDA's default lazy module loading, during the first
 *   gdn_prefill_noalloc call on that device -- and stays until the process
 *   exits, so a caller whose memory is fixed up front makes that first call in
 *   its set-up.
 *   A sequence layout needing more (gdn_prefill_workspace_size) is refused
 *   with GDN_ERR_WORKSPACE and nothing is enqueued; at Hk=16, Hv=32,
 *   d_k=d_v=128 the limit is a few hundred tokens per call.
 *   No call allocates: the first call on a device looks up the array's
 *   device address (cudaGetSymbolAddress) with that device current, so make
 *   that first call before any stream capture begins.  The address is kept
 *   per device for the life of the process; a cudaDeviceReset voids it.
 *   Every call on a device shares the one array: calls that can overlap on
 *   the GPU (on different streams, or from different threads without an
 *   ordering between them) race and give wrong results.  Calls ordered on one
 *   stream are safe; each call writes every scratch region it reads, so the
 *   previous call's contents never need clearing.
 */
gdn_status gdn_prefill_noalloc(const gdn_dims* dims, const gdn_params* params, int32_t n_seq,
                               const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                               const void* x, const void* z, const void* a, const void* b,
                               const void* conv_state_in, void* conv_state_out,
                               const float* initial_state, float* final_state, void* out,
                               void* stream);

/* Bytes of the built-in scratch array of gdn_prefill_noalloc. */
size_t gdn_prefill_noalloc_scratch_bytes(void);

/*
 * gdn_decode -- T tokens (1 <= T <= 16) for each of n_seq sequences against a
 * resident fp32 state: cpu.rs deltanet (one token) run T times, or a short
 * speculative-verify chunk.  Layouts are [n_seq, T, ...] (packed with uniform
 * lengths).  conv_state, when given, must be 16-byte aligned.
 *   inter_states == NULL: state [N, Hv, dk, dv] and conv_state [N, CD, K-1]
 *     are updated in place to their values after the T tokens.
 *   inter_states != NULL ([N, T, Hv, dk, dv]): the state after every token is
 *     written there and state and conv_state are only read, so the caller
 *     can keep any accepted prefix (gdn_decode_commit does that on the GPU).
 *   conv_state may be NULL (zero history, nothing written).
 */
gdn_status gdn_decode(const gdn_dims* dims, const gdn_params* params, int32_t n_seq,
                      int32_t T, const void* x, const void* z, const void* a, const void* b,
                      float* state, void* conv_state, float* inter_states, void* out,
                      void* stream);

/*
 * gdn_verify -- speculative verify for rollback by replay (qwen.rs
 * QwenSession::rewind keeps the pre-verify state and the drafts' inputs and
 * re-runs the accepted ones).  T draft tokens (1 <= T <= 16) of each sequence
 * run against state [N, Hv, dk, dv] and conv_state [N, CD, K-1] (may be NULL:
 * zero history), which are only read; out [N, T, Hv*dv] is the only write, so
 * the state traffic is one read.  Layouts as gdn_decode.  After acceptance
 * the caller replays each sequence's accepted prefix with gdn_prefill from the
 * same state and history (cu_seqlens built from the accepted counts; a prefix
 * of at most 16 tokens runs on the token-recurrent kernel), which writes the
 * new state and history.  Against gdn_decode with inter_states plus
 * gdn_decode_commit this moves (1 + 2) instead of (1 + T + 2) state slabs per
 * sequence, at the price of recomputing the accepted tokens.
 */
gdn_status gdn_verify(const gdn_dims* dims, const gdn_params* params, int32_t n_seq, int32_t T,
                      const void* x, const void* z, const void* a, const void* b,
                      const float* state, const void* conv_state, void* out, void* stream);

/*
 * gdn_decode_commit -- after a verify call of gdn_decode that wrote
 * inter_states, keep the first accepted[i] of the T tokens of sequence i:
 * state[i] becomes inter_states[i, accepted[i]-1] (left as is when
 * accepted[i] == 0) and conv_state[i] the last K-1 raw inputs of
 * (old history ++ x[i, :accepted[i]]).  This is the rewind of qwen.rs
 * QwenSession::rewind, done by selecting a kept state instead of replaying.
 *   accepted [n_seq] int32 device array; values are clamped to [0, T].
 *   x is the [n_seq, T, CD] input of the verify call; conv_state may be NULL.
 */
gdn_status gdn_decode_commit(const gdn_dims* dims, int32_t n_seq, int32_t T,
                             const int32_t* accepted, const void* x,
                             const float* inter_states, float* state, void* conv_state,
                             void* stream);

/* Weights of the projections around the core (a GDN layer's in_proj_* and
 * out_proj), bf16 device arrays in the [out_features, in_features] row-major
 * layout of qwen.rs's linear weights, 16-byte aligned. */
typedef struct gdn_proj {
    const void* w_qkv; /* [CD, hidden]    in_proj_qkv -> x */
    const void* w_z;   /* [Hv*dv, hidden] in_proj_z   -> z */
    const void* w_a;   /* [Hv, hidden]    in_proj_a   -> a */
    const void* w_b;   /* [Hv, hidden]    in_proj_b   -> b */
    const void* w_out; /* [hidden, Hv*dv] out_proj */
} gdn_proj;

/*
 * gdn_layer_prefill_workspace_size / gdn_layer_prefill -- one GDN layer's
 * prefill: the input projections x = h W_qkv^T, z = h W_z^T, a = h W_a^T,
 * b = h W_b^T (qwen.rs gdn_forward, its linear_multi over the hidden states),
 * the core exactly as gdn_prefill, then h_out = y W_out^T (out_proj).  bf16
 * only.  The projections run on this library's tcgen05 GEMM (bf16 operands,
 * fp32 accumulation): the four input projections in one launch that writes x,
 * z, a and b in the layouts the core reads, out_proj in a second.  Their
 * results, like the core's output y, are rounded to bf16, the core's
 * activation type.
 *   hidden: model width, a multiple of 8.  h_in, h_out [T, hidden] bf16.
 *   The states, cu_seqlens and their rules are those of gdn_prefill.
 *   workspace: at least gdn_layer_prefill_workspace_size() bytes, 256-byte
 *   aligned; it holds x, z, a, b, y and the core's workspace.
 */
gdn_status gdn_layer_prefill_workspace_size(const gdn_dims* dims, int32_t hidden, int32_t n_seq,
                                            const int32_t* cu_seqlens_host, size_t* bytes);
gdn_status gdn_layer_prefill(const gdn_dims* dims, const gdn_params* params,
                             const gdn_proj* proj, int32_t hidden, int32_t n_seq,
                             const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                             const void* h_in, const float* initial_state, float* final_state,
                             const void* conv_state_in, void* conv_state_out, void* h_out,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_timing_enable / gdn_timing_report -- per-kernel device timing (the
 * library's tracing hook; the pages time their GDN phases with scoped timers,
 * qwen.rs gdn_forward prof::start).  While enabled, every kernel launch the
 * library makes is bracketed by CUDA events recorded on its stream.
 *   gdn_timing_enable(1) clears the totals and starts recording; (0) stops.
 *   gdn_timing_report waits for the recorded events, then writes one line per
 *   kernel, "<name> <launches> <total_ms>\n", into buf (NUL-terminated,
 *   truncated to buf_len) and returns the bytes the full report needs.
 * Process-wide; thread-safe; not for use while a CUDA graph is captured.
 */
gdn_status gdn_timing_enable(int32_t enable);
size_t gdn_timing_report(char* buf, size_t buf_len);

/*
 * gdn_device_error -- the library's sticky device-side error word.  Kernels
 * whose waits are bounded (the tensor-core prefill waits on its own TMA copies
 * and MMAs) give up after ~2 s instead of hanging, store a nonzero code here
 * (1..12 name the tensor-core prefill's wait that gave up, 11 being a fused
 * launch's wait for a chunk's prep rows; 13 and 14 its per-channel decay prep's
 * waits for its tiles, and for its v tile, products and the next item's tiles;
 * 20..23 the projection GEMM's; 30 the
 * token-recurrent kernel's wait for a state copy) and exit cleanly; their
 * outputs are then invalid.  Waits for the device (cudaMemcpyFromSymbol), writes the code to
 * *code (0 = no error) and clears it when reset != 0.
 */
gdn_status gdn_device_error(int32_t* code, int32_t reset);

/*
 * gdn_sync_status -- waits for `stream` (cudaStream_t as void*), then reads and
 * clears the device error word: GDN_ERR_TIMEOUT if a bounded device wait gave
 * up since the last check (the outputs and states of the calls since then are
 * invalid and must be recomputed; the CUDA context stays usable), GDN_ERR_CUDA
 * if the stream reports a CUDA error, else GDN_OK.  A serving loop calls it
 * where it would synchronize anyway, and fails the affected requests closed.
 */
gdn_status gdn_sync_status(void* stream);

/* Message for the last failed call on this thread ("" if none). */
const char* gdn_last_error(void);

/* Library version string. */
const char* gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
