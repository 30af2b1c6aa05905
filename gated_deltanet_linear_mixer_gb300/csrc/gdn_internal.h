// Internal launch interface between the C-ABI layer (gdn_api.cu) and the
// kernels.  Host-visible plain structs; pointers are device pointers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct ConvArgs {
    int n_seq, n_tokens, n_k_heads, n_v_heads, d_k, d_v, conv_k;
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
    float* g_out;               // [T, Hv]
    float* beta_out;            // [T, Hv]
};

struct ConvStateArgs {
    int n_seq, n_k_heads, n_v_heads, d_k, d_v, conv_k;
    const int32_t* cu_seqlens;  // [n_seq+1], or null with uniform_T tokens per sequence
    int uniform_T;
    const int32_t* lengths;     // optional per-sequence prefix length (commit), or null
    const void* x;
    const void* conv_state_in;  // or null (zeros)
    void* conv_state_out;
};

struct RecurrentArgs {
    int n_seq, n_k_heads, n_v_heads, conv_k, act;
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

cudaError_t launch_conv_prologue(const ConvArgs& p, bool bf16, cudaStream_t stream);
cudaError_t launch_conv_state(const ConvStateArgs& p, bool bf16, cudaStream_t stream);
cudaError_t launch_recurrent(const RecurrentArgs& p, int d_k, int d_v, bool bf16,
                             cudaStream_t stream);
cudaError_t launch_commit_state(const CommitArgs& p, cudaStream_t stream);

}  // namespace gdn
