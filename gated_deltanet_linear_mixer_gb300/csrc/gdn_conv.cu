// Prologue kernels of the GDN core: causal depthwise conv + SiLU, q/k L2
// normalisation with the q scale, the decay/write gates, and the conv-state
// update (oxinfer 0.0.5 src/qwen.rs, fn gdn_forward and DeltaRule::run;
// cherenkov qwen4_exp/cpu.rs, fn causal_conv).
//
// Work split: one CTA = one head's channels ("unit": a q head, a k head or a
// v head) x a tile of 64 tokens.  Each thread owns one 16-byte vector of
// channels (8 bf16 / 4 fp32) and a run of consecutive tokens; it loads each
// raw row of its window once (all loads issued up front), so loads and stores
// of x and qkv_out are 16-byte and coalesced; the d-wide L2 norm of a q/k head
// is a shuffle reduction over the d/VEC lanes that share the token.  One extra
// unit per token tile computes g and beta.  The whole pass reads x once and
// writes qkv_out once, so it is bound by HBM bandwidth.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kConvThreads = 128;

// Channel ch of sequence n (first token bos, len tokens): its new history is
// the last K-1 raw inputs, oldest first, shifted in from the old history when
// the sequence is shorter than K-1 (zeros without one).
template <typename T>
__device__ __forceinline__ void conv_history_one(const T* __restrict__ x, const T* __restrict__ cs_in,
                                                 T* __restrict__ cs_out, int cd, int keep, int n,
                                                 int ch, int bos, int len) {
    T nw[3];
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (s >= keep) break;
        const int ti = len - keep + s;
        if (ti >= 0)
            nw[s] = x[(size_t)(bos + ti) * cd + ch];
        else if (cs_in)
            nw[s] = cs_in[((size_t)n * cd + ch) * keep + keep + ti];
        else
            nw[s] = from_f32<T>(0.0f);
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        if (s >= keep) break;
        cs_out[((size_t)n * cd + ch) * keep + s] = nw[s];
    }
}
constexpr int kConvTokTile = 64;

template <typename T>
__global__ void __launch_bounds__(kConvThreads)
conv_prologue_kernel(ConvArgs p) {
    using V = Vec16<T>;
    constexpr int VEC = V::N;
    const int n_units = 2 * p.n_k_heads + p.n_v_heads;
    const int unit = blockIdx.y;
    const int tile0 = blockIdx.x * kConvTokTile;
    const int cd = 2 * p.n_k_heads * p.d_k + p.n_v_heads * p.d_v;
    const T* __restrict__ x = static_cast<const T*>(p.x);

    if (unit == n_units) {  // gates for this token tile
        const int hv_n = p.n_v_heads;
        const T* __restrict__ a = static_cast<const T*>(p.a);
        const T* __restrict__ b = static_cast<const T*>(p.b);
        const int nc = p.per_channel ? p.d_k : 1;  // decays per value head
        for (int i = threadIdx.x; i < kConvTokTile * hv_n * nc; i += kConvThreads) {
            const int t = tile0 + i / (hv_n * nc);
            const int h = (i / nc) % hv_n, j = i % nc;
            if (t >= p.n_tokens) break;
            const size_t idx = (size_t)t * hv_n + h;
            p.g_out[idx * nc + j] = log_decay(to_f32(a[idx * nc + j]), p.A_log[h],
                                              p.dt_bias[(size_t)h * nc + j], p.decay_form);
            if (j == 0) p.beta_out[idx] = sigmoidf_(to_f32(b[idx]));
        }
        return;
    }

    const bool is_q = unit < p.n_k_heads;
    const bool is_k = !is_q && unit < 2 * p.n_k_heads;
    const int D = (is_q || is_k) ? p.d_k : p.d_v;
    const int ch0 = (is_q || is_k) ? unit * p.d_k
                                   : 2 * p.n_k_heads * p.d_k + (unit - 2 * p.n_k_heads) * p.d_v;
    const int tpr = D / VEC;                 // threads per token row (power of 2, <= 32)
    const int runs = kConvThreads / tpr;     // token runs per tile
    const int TR = kConvTokTile / runs;      // consecutive tokens per thread (2..16)
    const int lane_in_row = threadIdx.x % tpr;
    const int run = threadIdx.x / tpr;
    const int c = ch0 + lane_in_row * VEC;   // first channel of this thread
    const int K = p.conv_k;
    const int keep = K - 1;
    const int tr0 = tile0 + run * TR;        // first token of this thread's run

    // Taps padded to 4 with leading zero weights: padded tap k multiplies
    // raw row t-3+k, so every window index below is a compile-time constant.
    const int pad = 4 - K;
    float w[VEC][4];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[e][k] = k >= pad ? p.conv_w[(size_t)(c + e) * K + (k - pad)] : 0.0f;

    const float qscale = rsqrtf((float)p.d_k);
    const T* __restrict__ cs_in = static_cast<const T*>(p.conv_state_in);
    T* __restrict__ out = static_cast<T*>(p.qkv_out);
    T* __restrict__ out_lo = static_cast<T*>(p.qkv_lo_out);

    // Sliding window in passes of up to 8 tokens: the raw rows t-3 .. t+7 of a
    // pass are loaded once each, all issued before any is used.
    constexpr int kPass = 8;
    for (int p0 = 0; p0 < TR; p0 += kPass) {
        const int tp = tr0 + p0;
        uint4 raw[kPass + 3];  // packed rows, unpacked at use
#pragma unroll
        for (int i = 0; i < kPass + 3; ++i) {
            const int row = tp - 3 + i;
            raw[i] = (i < TR - p0 + 3 && row >= 0 && row < p.n_tokens)
                         ? V::load_raw(x + (size_t)row * cd + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        int n = 0, bos = 0, eos = 0;
        if (tp < p.n_tokens) {
            n = seq_of_token(p.cu_seqlens, p.n_seq, tp);
            bos = p.cu_seqlens[n];
            eos = p.cu_seqlens[n + 1];
        }
#pragma unroll
        for (int j = 0; j < kPass; ++j) {
            if (p0 + j >= TR) break;  // uniform across the warp: TR is per CTA
            const int t = tp + j;
            const bool valid = t < p.n_tokens;
            if (valid) {
                while (t >= eos) {  // crossed into the next non-empty sequence
                    ++n;
                    bos = p.cu_seqlens[n];
                    eos = p.cu_seqlens[n + 1];
                }
            }
            float acc[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
            if (valid) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (k < pad) continue;
                    const int src = t - 3 + k;           // raw row j + k of the window
                    if (src >= bos) {
                        float v[VEC];
                        V::unpack(raw[j + k], v);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w[e][k], v[e], acc[e]);
                    } else if (cs_in) {
                        const int slot = keep + (src - bos);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            acc[e] = fmaf(w[e][k], to_f32(cs_in[((size_t)n * cd + c + e) * keep + slot]),
                                          acc[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = siluf_(acc[e]);
            }
            if (is_q || is_k) {
                float ss = 0.0f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) ss = fmaf(acc[e], acc[e], ss);
                for (int off = tpr / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                float inv = rsqrtf(ss + p.l2_eps);
                if (is_q) inv *= qscale;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] *= inv;
            }
            if (valid) {
                V::store(out + (size_t)t * cd + c, acc);
                if (out_lo) {  // bf16 residual: acc = hi + lo to ~16 significant bits
                    float lo[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) lo[e] = acc[e] - to_f32(from_f32<T>(acc[e]));
                    V::store(out_lo + (size_t)t * cd + c, lo);
                }
            }
        }
    }
}

// cu_chunks[i] = sum over sequences j < i of ceil(len_j / C); per chunk its
// first token and length; the item flags cleared.  One CTA of 256 threads.
__device__ void chunk_table_cta(const ConvArgs& p) {
    __shared__ int32_t warp_tot[8];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < p.n_ready; i += 256) p.ready[i] = 0;
    if (tid == 0) {
        carry = 0;
        p.cu_chunks[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < p.n_seq; base += 256) {
        const int i = base + tid;
        const int v = i < p.n_seq ? (p.cu_seqlens[i + 1] - p.cu_seqlens[i] + kChunkTokens - 1) / kChunkTokens : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < 8 ? warp_tot[lane] : 0;
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            if (lane < 8) warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + carry;
        if (i < p.n_seq) p.cu_chunks[i + 1] = before + incl;
        __syncthreads();
        if (tid == 255) carry = before + incl;
        __syncthreads();
    }
    const int n_chunks = p.n_seq > 0 ? p.cu_chunks[p.n_seq] : 0;
    if (p.seq_order) {  // rank of sequence i: longer ones first, ties in index order
        for (int i = tid; i < p.n_seq; i += 256) {
            const int ci = p.cu_chunks[i + 1] - p.cu_chunks[i];
            int rank = 0;
            for (int j = 0; j < p.n_seq; ++j) {
                const int cj = p.cu_chunks[j + 1] - p.cu_chunks[j];
                rank += cj > ci || (cj == ci && j < i);
            }
            p.seq_order[rank] = i;
        }
    }
    for (int c = tid; c < n_chunks; c += 256) {
        const int n = seq_of_token(p.cu_chunks, p.n_seq, c);
        const int t0 = p.cu_seqlens[n] + (c - p.cu_chunks[n]) * kChunkTokens;
        p.chunk_info[c] = make_int2(t0, min(kChunkTokens, p.cu_seqlens[n + 1] - t0));
    }
}

// The prologue for bf16 activations with d_k = d_v = 128 (the tensor-core
// prefill): one warp per (128-channel unit, 8-token run), 4 channels per lane,
// four CTAs per SM.  The warp's 11 raw rows (3 of halo) are loaded up front with 8-byte
// coalesced loads; per token the L2 norm of a q/k head is a full-warp
// reduction.  Writes q|k|v as a (hi, lo) bf16 pair, g and beta like
// conv_prologue_kernel; the first CTA of the gate row also builds the chunk table.
// With per-channel decay the gate row writes only beta (the chunked prep forms
// the decays from a itself).
constexpr int kPro128Tok = 8;                   // tokens per warp
constexpr int kPro128Tile = 8 * kPro128Tok;     // tokens per CTA

__global__ void __launch_bounds__(256, 4) conv_prologue_d128_kernel(ConvArgs p) {
    const int n_units = 2 * p.n_k_heads + p.n_v_heads;
    const int unit = blockIdx.y;
    const int tile0 = blockIdx.x * kPro128Tile;
    const int cd = n_units * 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const __nv_bfloat16* __restrict__ x = static_cast<const __nv_bfloat16*>(p.x);

    if (unit == n_units + 1) {  // the new conv history of every sequence (grid-stride)
        const int keep = p.conv_k - 1;
        const int nblk = (cd + 255) / 256;
        for (int it = blockIdx.x; it < p.n_seq * nblk; it += gridDim.x) {
            const int n = it / nblk, ch = (it % nblk) * 256 + tid;
            if (ch < cd)
                conv_history_one<__nv_bfloat16>(x, static_cast<const __nv_bfloat16*>(p.conv_state_in),
                                                static_cast<__nv_bfloat16*>(p.conv_state_out), cd, keep,
                                                n, ch, p.cu_seqlens[n], p.cu_seqlens[n + 1] - p.cu_seqlens[n]);
        }
        return;
    }
    if (unit == n_units) {  // gates for this token tile (and, in the first, the chunk table)
        if (blockIdx.x == 0 && p.cu_chunks) chunk_table_cta(p);
        const int hv_n = p.n_v_heads;
        const __nv_bfloat16* __restrict__ a = static_cast<const __nv_bfloat16*>(p.a);
        const __nv_bfloat16* __restrict__ b = static_cast<const __nv_bfloat16*>(p.b);
        for (int i = tid; i < kPro128Tile * hv_n; i += 256) {
            const int t = tile0 + i / hv_n;
            const int h = i % hv_n;
            if (t >= p.n_tokens) break;
            const size_t idx = (size_t)t * hv_n + h;
            if (!p.per_channel)
                p.g_out[idx] = log_decay(__bfloat162float(a[idx]), p.A_log[h], p.dt_bias[h], p.decay_form);
            p.beta_out[idx] = sigmoidf_(__bfloat162float(b[idx]));
        }
        return;
    }
    const int tb = tile0 + warp * kPro128Tok;  // first token of this warp
    const int c = unit * 128 + 4 * lane;       // first channel of this lane
    __nv_bfloat16* __restrict__ out = static_cast<__nv_bfloat16*>(p.qkv_out);
    __nv_bfloat16* __restrict__ out_lo = static_cast<__nv_bfloat16*>(p.qkv_lo_out);
    for (int t = max(tb, p.n_tokens); t < min(tb + kPro128Tok, p.n_tokens + p.zero_tail); ++t) {
        *reinterpret_cast<uint2*>(out + (size_t)t * cd + c) = make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(out_lo + (size_t)t * cd + c) = make_uint2(0u, 0u);
    }
    if (tb >= p.n_tokens) return;              // warp-uniform
    const bool is_q = unit < p.n_k_heads;
    const bool norm = unit < 2 * p.n_k_heads;
    const float scale = is_q ? rsqrtf(128.f) : 1.f;
    const int K = p.conv_k, keep = K - 1, pad = 4 - K;
    float w[4][4];
    if (K == 4 && (reinterpret_cast<uintptr_t>(p.conv_w) & 15u) == 0) {  // 4 channels x 4 taps, 64 B
        const float4* wp = reinterpret_cast<const float4*>(p.conv_w + (size_t)c * 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 v = wp[e];
            w[e][0] = v.x; w[e][1] = v.y; w[e][2] = v.z; w[e][3] = v.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int k = 0; k < 4; ++k) w[e][k] = k >= pad ? p.conv_w[(size_t)(c + e) * K + (k - pad)] : 0.f;
    }
    uint2 raw[kPro128Tok + 3];  // rows tb-3 .. tb+7
#pragma unroll
    for (int i = 0; i < kPro128Tok + 3; ++i) {
        const int rr = tb - 3 + i;
        raw[i] = (rr >= 0 && rr < p.n_tokens) ? *reinterpret_cast<const uint2*>(x + (size_t)rr * cd + c)
                                              : make_uint2(0u, 0u);
    }
    const __nv_bfloat16* __restrict__ cs_in = static_cast<const __nv_bfloat16*>(p.conv_state_in);
    int n = seq_of_token(p.cu_seqlens, p.n_seq, tb);
    int bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    // SiLU, the q/k L2 norm (q scaled), the (hi, lo) split and the stores of token t
    auto finish = [&](float* acc, int t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = siluf_(acc[e]);
        if (norm) {
            float ss = acc[0] * acc[0] + acc[1] * acc[1] + acc[2] * acc[2] + acc[3] * acc[3];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss + p.l2_eps) * scale;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] *= inv;
        }
        const uint32_t h01 = pack_bf16_pair(acc[0], acc[1]), h23 = pack_bf16_pair(acc[2], acc[3]);
        const float l0 = acc[0] - __uint_as_float(h01 << 16), l1 = acc[1] - __uint_as_float(h01 & 0xFFFF0000u);
        const float l2 = acc[2] - __uint_as_float(h23 << 16), l3 = acc[3] - __uint_as_float(h23 & 0xFFFF0000u);
        *reinterpret_cast<uint2*>(out + (size_t)t * cd + c) = make_uint2(h01, h23);
        *reinterpret_cast<uint2*>(out_lo + (size_t)t * cd + c) =
            make_uint2(pack_bf16_pair(l0, l1), pack_bf16_pair(l2, l3));
    };
    if (tb - 3 >= bos && tb + kPro128Tok <= eos) {  // the run and its halo lie in one sequence
#pragma unroll
        for (int j = 0; j < kPro128Tok; ++j) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint2 r = raw[j + k];
                acc[0] = fmaf(w[0][k], __uint_as_float(r.x << 16), acc[0]);
                acc[1] = fmaf(w[1][k], __uint_as_float(r.x & 0xFFFF0000u), acc[1]);
                acc[2] = fmaf(w[2][k], __uint_as_float(r.y << 16), acc[2]);
                acc[3] = fmaf(w[3][k], __uint_as_float(r.y & 0xFFFF0000u), acc[3]);
            }
            finish(acc, tb + j);
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < kPro128Tok; ++j) {
        const int t = tb + j;
        if (t >= p.n_tokens) break;  // warp-uniform
        while (t >= eos) {           // crossed into the next non-empty sequence
            ++n;
            bos = p.cu_seqlens[n];
            eos = p.cu_seqlens[n + 1];
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int src = t - 3 + k;
            float v[4];
            if (src >= bos) {
                const uint2 r = raw[j + k];
                v[0] = __uint_as_float(r.x << 16); v[1] = __uint_as_float(r.x & 0xFFFF0000u);
                v[2] = __uint_as_float(r.y << 16); v[3] = __uint_as_float(r.y & 0xFFFF0000u);
            } else if (cs_in && src >= bos - keep) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v[e] = __bfloat162float(cs_in[((size_t)n * cd + c + e) * keep + keep + (src - bos)]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(w[e][k], v[e], acc[e]);
        }
        finish(acc, t);
    }
}

// New history of each sequence = its last K-1 raw inputs, oldest first,
// shifted in from the old history when the sequence is shorter than K-1.
template <typename T>
__global__ void conv_state_kernel(ConvStateArgs p) {
    const int n = blockIdx.y;
    const int ch = blockIdx.x * blockDim.x + threadIdx.x;
    const int cd = 2 * p.n_k_heads * p.d_k + p.n_v_heads * p.d_v;
    if (ch >= cd) return;
    const int keep = p.conv_k - 1;
    int bos, len;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - bos;
    } else {
        bos = n * p.uniform_T;
        len = p.uniform_T;
    }
    if (p.lengths) len = min(max(p.lengths[n], 0), len);  // accepted prefix (commit)
    conv_history_one<T>(static_cast<const T*>(p.x), static_cast<const T*>(p.conv_state_in),
                        static_cast<T*>(p.conv_state_out), cd, keep, n, ch, bos, len);
}

cudaError_t launch_conv_prologue(const ConvArgs& p, bool bf16, cudaStream_t stream) {
    if (p.n_tokens == 0) return cudaSuccess;
    if (bf16 && p.d_k == 128 && p.d_v == 128 && p.qkv_lo_out) {
        dim3 grid((p.n_tokens + p.zero_tail + kPro128Tile - 1) / kPro128Tile,
                  2 * p.n_k_heads + p.n_v_heads + 1 + (p.conv_state_out ? 1 : 0));
        conv_prologue_d128_kernel<<<grid, 256, 0, stream>>>(p);
        return cudaGetLastError();
    }
    dim3 grid((p.n_tokens + kConvTokTile - 1) / kConvTokTile, 2 * p.n_k_heads + p.n_v_heads + 1);
    if (bf16)
        conv_prologue_kernel<__nv_bfloat16><<<grid, kConvThreads, 0, stream>>>(p);
    else
        conv_prologue_kernel<float><<<grid, kConvThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// The same for K = 4 (three history slots), 16 bytes of channels a thread: its
// history block (3 x 16 bytes, slot-minor) is read and written whole, and each
// new input row is one 16-byte load.  A thread reads and writes only its own
// block, so the update may be in place.
template <typename T>
__global__ void conv_state_vec_kernel(ConvStateArgs p) {
    constexpr int VEC = 16 / (int)sizeof(T);  // channels a thread
    constexpr int KEEP = 3;
    const int n = blockIdx.y;
    const int cd = 2 * p.n_k_heads * p.d_k + p.n_v_heads * p.d_v;
    const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * VEC;
    if (c0 >= cd) return;
    int bos, len;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - bos;
    } else {
        bos = n * p.uniform_T;
        len = p.uniform_T;
    }
    if (p.lengths) len = min(max(p.lengths[n], 0), len);  // accepted prefix (commit)
    const T* __restrict__ x = static_cast<const T*>(p.x);
    const size_t blk = ((size_t)n * cd + c0) * KEEP;  // element offset of the block
    union Block { uint4 u[KEEP]; T v[KEEP * VEC]; };
    Block old, nw;
    if (len < KEEP) {  // some slots come from the old history (zeros without one)
        if (p.conv_state_in) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.conv_state_in) + blk);
#pragma unroll
            for (int i = 0; i < KEEP; ++i) old.u[i] = src[i];
        } else {
#pragma unroll
            for (int i = 0; i < KEEP; ++i) old.u[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int s = 0; s < KEEP; ++s) {
        const int ti = len - KEEP + s;  // token of slot s, relative to the sequence start
        if (ti >= 0) {
            union { uint4 u; T v[VEC]; } row;
            row.u = *reinterpret_cast<const uint4*>(x + (size_t)(bos + ti) * cd + c0);
#pragma unroll
            for (int e = 0; e < VEC; ++e) nw.v[e * KEEP + s] = row.v[e];
        } else {  // old slot j = KEEP + ti (0..2), picked with constant indices
            const int j = KEEP + ti;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                nw.v[e * KEEP + s] = j == 0 ? old.v[e * KEEP] : (j == 1 ? old.v[e * KEEP + 1] : old.v[e * KEEP + 2]);
        }
    }
    // a programmatic dependent stores only once the preceding grid, which may
    // still read the old history, has completed
    if (p.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.conv_state_out) + blk);
#pragma unroll
    for (int i = 0; i < KEEP; ++i) dst[i] = nw.u[i];
}

cudaError_t launch_conv_state(const ConvStateArgs& p, bool bf16, cudaStream_t stream) {
    if (p.n_seq == 0 || p.conv_k < 2) return cudaSuccess;
    const int cd = 2 * p.n_k_heads * p.d_k + p.n_v_heads * p.d_v;
    const int vec = bf16 ? 8 : 4;
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    if (p.conv_k == 4 && cd % vec == 0 && al16(p.x) && al16(p.conv_state_out) &&
        (!p.conv_state_in || al16(p.conv_state_in))) {
        dim3 grid((cd / vec + 255) / 256, p.n_seq);
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        if (p.pdl) {
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
        }
        return bf16 ? cudaLaunchKernelEx(&cfg, conv_state_vec_kernel<__nv_bfloat16>, p)
                    : cudaLaunchKernelEx(&cfg, conv_state_vec_kernel<float>, p);
    }
    dim3 grid((cd + 255) / 256, p.n_seq);
    if (bf16)
        conv_state_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(p);
    else
        conv_state_kernel<float><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
