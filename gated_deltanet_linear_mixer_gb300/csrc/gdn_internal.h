// Internal launch interface between the C-ABI layer (gdn_api.cu) and the
// kernels.  Host-visible plain structs; pointers are device pointers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Tokens per chunk of the tensor-core prefill.
constexpr int kChunkTokens = 64;

struct ConvArgs {
    int n_seq, n_tokens, n_k_heads, n_v_heads, d_k, d_v, conv_k;
    int decay_form;             // gdn_decay_form
    int per_channel;            // one decay per key channel: a [T, Hv*dk], g_out [T, Hv*dk]
                                //   (the d=128 prologue writes only beta then: the
                                //   chunked prep forms g itself)
    float l2_eps;
    const int32_t* cu_seqlens;  // [n_seq+1]
    const void* x;              // [T, CD]
    const void* a;              // [T, Hv]
    const void* b;              // [T, Hv]
    const float* conv_w;        // [CD, K]
    const float* A_log;         // [Hv]
    const float* dt_bias;       // [Hv]
    const void* conv_state_in;  // [N, CD, K-1] or null
    void* qkv_out;              // [T, CD]
    void* qkv_lo_out;           // [T, CD] bf16 residual x - bf16(x), or null (bf16 only)
    float* g_out;               // [T, Hv]
    float* beta_out;            // [T, Hv]
    int zero_tail;              // rows [T, T + zero_tail) of qkv_out / qkv_lo_out set to 0
    // Chunk table of the tensor-core prefill, built by one CTA of the d=128
    // prologue (null otherwise): offsets per sequence, (first token, length)
    // per chunk, and n_ready item flags cleared.
    int32_t* cu_chunks;         // [n_seq+1]
    int2* chunk_info;           // [chunks]
    int* ready;
    int n_ready;
    int32_t* seq_order;         // [n_seq] sequences by chunk count, longest first, or null
    // New conv history [N, CD, K-1], written by an extra CTA row of the d=128
    // prologue; only when it does not alias conv_state_in (else null)
    void* conv_state_out;
};

struct ConvStateArgs {
    int n_seq, n_k_heads, n_v_heads, d_k, d_v, conv_k;
    const int32_t* cu_seqlens;  // [n_seq+1], or null with uniform_T tokens per sequence
    int uniform_T;
    const int32_t* lengths;     // optional per-sequence prefix length (commit), or null
    const void* x;
    const void* conv_state_in;  // or null (zeros)
    void* conv_state_out;
    // Launched as the programmatic dependent of the preceding kernel (which may
    // let it start early): its loads come first, its stores after that kernel
    // has completed.
    int pdl;
};

struct RecurrentArgs {
    int n_seq, n_k_heads, n_v_heads, conv_k, act;
    int head_map, decay_form;   // gdn_head_map, gdn_decay_form
    int per_channel;            // one decay per key channel (a [T, Hv*dk], dt_bias [Hv*dk])
    float l2_eps, rms_eps;
    const int32_t* cu_seqlens;  // [n_seq+1], or null with uniform_T tokens per sequence
    int uniform_T;
    const void* x;              // [T, CD]
    const void* z;              // [T, Hv*dv]
    const void* a;
    const void* b;
    const float* conv_w;
    const float* A_log;
    const float* dt_bias;
    const float* norm_w;
    const void* conv_state_in;  // or null
    const float* state_in;      // [N, Hv, dk, dv] or null (zeros)
    float* state_out;           // or null; may equal state_in
    float* inter;               // [T, Hv, dk, dv] or null
    void* out;                  // [T, Hv*dv]
};

struct CommitArgs {
    int n_seq, n_v_heads, d_k, d_v, T;
    const int32_t* accepted;  // [n_seq]
    const float* inter;       // [n_seq, T, Hv, dk, dv]
    float* state;             // [n_seq, Hv, dk, dv]
};

// Arguments of the chunked (tensor-core) kernels.  Operands that feed the
// tensor cores are kept as bf16 (hi, lo) pairs: hi = bf16(x), lo = bf16(x - hi).
struct ChunkArgs {
    int n_seq, n_tokens, n_chunks, n_k_heads, n_v_heads, act;
    int head_map;                 // gdn_head_map
    float rms_eps;
    const int32_t* cu_seqlens;    // [n_seq+1]
    const int32_t* cu_chunks;     // [n_seq+1] chunk offsets (workspace)
    const int2* chunk_info;       // [chunks] first token and length of each chunk (workspace)
    const int32_t* seq_order;     // [n_seq] scan launch order (longest first), or null
    const __nv_bfloat16* qkv_hi;  // [T, CD] normalised q | k | v, hi part (workspace)
    const __nv_bfloat16* qkv_lo;  // [T, CD] lo part (workspace)
    const float* g;               // [T, Hv] log-decay (workspace; not with per-channel decay)
    const float* beta;            // [T, Hv] (workspace)
    const __nv_bfloat16* z;       // [T, Hv*dv]
    const float* norm_w;          // [dv]
    const float* state_in;        // [N, Hv, dk, dv] or null
    float* state_out;             // or null
    __nv_bfloat16* w_hi;          // [chunks, Hv, 64, dk] W (hi, lo); per-channel decay: then
    __nv_bfloat16* w_lo;          //   Q o e^G in the same layout from row qt_row0 on
    int qt_row0;                  // chunks * Hv * 64 (per-channel decay), else 0
    // Per-channel decay: its prep forms g = coef softplus(a + dt_bias) itself
    // from the raw gate input (the prologue writes only beta).
    const __nv_bfloat16* gate_a;  // [T, Hv*dk] (read through a tensor map: 16-byte aligned)
    const float* A_log;           // [Hv] (or the coefficient, decay_form)
    const float* dt_bias;         // [Hv*dk]
    int decay_form;
    __nv_bfloat16* kw_hi;         // per-channel decay: [chunks, Hv, 64, dk] K o e^{G_last-G}
    __nv_bfloat16* kw_lo;         //   (hi, lo), written by its prep (else by TMA, unused here)
    float* u_ws;                  // [chunks, Hv, dv/4, 64, 4] U~ (fp32), 4-column groups
    __nv_bfloat16* qk_hi;         // [chunks, Hv, 64, 64] masked decayed Q K^T (hi, lo)
    __nv_bfloat16* qk_lo;
    float* gcum_ws;               // [chunks, Hv, 64] in-chunk cumulative log-decay; per-channel
                                  //   decay: [chunks, Hv, dk] G_last of each key channel
    __nv_bfloat16* out;           // [T, Hv*dv]
    int* ready;                   // [chunks, Hk] item done flags (fused launch), else null
    // Test hook (fused launch): when set, the scan waits on this flag, which
    // nothing sets, for at most wait_ns, so that its bounded wait runs out.
    const int* stall_flag;
    unsigned long long wait_ns;   // limit of the scan's wait for a chunk's prep rows
};

// Byte offsets of the chunked path's workspace regions.
struct ChunkLayout {
    size_t qkv_hi, qkv_lo, g, beta, cu_chunks, chunk_info, seq_order, w_hi, w_lo, u, qk_hi, qk_lo,
        kw_hi, kw_lo, gcum, ready, total;
    int n_chunks;
    int per_channel;
};

// Per-kernel timing hook (CUDA events on the launching stream when enabled).
void* timing_start(const char* name, cudaStream_t stream);
void timing_stop(void* handle, cudaStream_t stream);
template <typename F>
cudaError_t timed_launch(const char* name, cudaStream_t stream, F&& launch) {
    void* h = timing_start(name, stream);
    cudaError_t e = launch();
    timing_stop(h, stream);
    return e;
}

struct ChunkLaunch {
    int n_seq, n_tokens, n_k_heads, n_v_heads, conv_k, act;
    int head_map, decay_form;
    int per_channel;       // one decay per key channel (a [T, Hv*dk], dt_bias [Hv*dk])
    float l2_eps, rms_eps;
    const int32_t* cu_seqlens;
    const void *x, *z, *a, *b;
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    const void* conv_state_in;
    void* conv_state_out;  // written by the prologue when set (see ConvArgs)
    const float* state_in;
    float* state_out;
    void* out;
    void* workspace;
    ChunkLayout layout;
    int stall;             // test hook: the fused scan waits on a flag nothing sets
};

// Workspace size (and layout) of the chunked path for this sequence layout.
size_t chunked_workspace_bytes(int n_seq, const int32_t* cu_host, int n_k_heads, int n_v_heads,
                               int per_channel, ChunkLayout* layout);
// Whether the chunked tensor-core path serves this geometry.
inline bool chunked_supported(int d_k, int d_v, int n_k_heads, int n_v_heads, bool bf16) {
    return bf16 && d_k == 128 && d_v == 128 && n_v_heads / n_k_heads <= 8;
}
cudaError_t launch_chunked_prefill(const ChunkLaunch& a, cudaStream_t stream);
// The per-channel decay prep (gdn_chunked_kda.cu): n_ctas persistent CTAs over
// the (chunk, value head) items; the maps are the q|k|v (hi, lo) tiles and the
// M o QK^T rows (hi, lo) of the workspace, and the gate input a [T, Hv*128].
cudaError_t launch_kda_prep(const CUtensorMap& map_qh, const CUtensorMap& map_ql, const CUtensorMap& map_kqh,
                            const CUtensorMap& map_kql, const CUtensorMap& map_a, const ChunkArgs& p, int n_ctas,
                            cudaStream_t stream);
size_t kda_prep_smem_bytes();
cudaError_t read_kda_error(int* code, bool reset);
// Sticky device-side error word set by a kernel whose bounded wait gave up.
cudaError_t read_device_error(int* code, bool reset);

// Projection GEMM on tcgen05: C_s = A W_s^T for up to four weights W_s that
// share A (all bf16 row-major; W_s is [n, k], C_s is [m, n] with row stride
// ldc), one launch.  A, W_s and C_s 16-byte aligned; k a multiple of 8.
struct GemmSegment {
    const void* w;
    void* c;
    int n, ldc;
};
struct GemmLaunch {
    const void* a;
    int m, k, n_seg;
    GemmSegment seg[4];
};
cudaError_t launch_gemm_bf16(const GemmLaunch& g, cudaStream_t stream);
// The projection GEMM's device error word (a bounded wait that gave up).
cudaError_t read_gemm_error(int* code, bool reset);

cudaError_t launch_conv_prologue(const ConvArgs& p, bool bf16, cudaStream_t stream);
cudaError_t launch_conv_state(const ConvStateArgs& p, bool bf16, cudaStream_t stream);
cudaError_t launch_recurrent(const RecurrentArgs& p, int d_k, int d_v, bool bf16,
                             cudaStream_t stream);
cudaError_t launch_commit_state(const CommitArgs& p, cudaStream_t stream);
// The token-recurrent kernel's device error word (30: a state copy wait gave up).
cudaError_t read_rec_error(int* code, bool reset);

}  // namespace gdn
