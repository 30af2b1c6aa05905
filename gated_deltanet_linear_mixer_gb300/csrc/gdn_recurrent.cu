// Token-recurrent GDN kernel: the decode path (one or a few tokens per
// sequence against a resident fp32 state) and the fp32 prefill path.
//
// It runs the delta rule exactly as cherenkov qwen4_exp/cpu.rs fn deltanet
// and oxinfer 0.0.5 src/qwen.rs DeltaRule::run define it (decay, read of the
// decayed state, rank-one write, readout), with the conv/normalise/gate
// prologue and the gated-RMSNorm epilogue fused in.
//
// Design (memory-bound): one CTA of 256 threads per (sequence, value head).
// The d_k x d_v fp32 state slab is streamed from HBM once, held in registers
// for all the tokens of the call, and written back once.  Thread layout: a
// state row (d_v floats) is covered by d_v/4 lanes with one float4 each, so
// every load/store instruction of a warp moves whole 128..512-byte rows; the
// CTA's row groups split the d_k rows.  The two per-token column reductions
// S^T k and S^T q share one pass: warp shuffles across the row groups inside
// a warp, then shared memory across warps.  The readout uses
// o = e^g S^T q + (k.q) delta, which equals S'^T q for the written state S'
// (S' = e^g S + k delta^T), so the state is read once per token.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kRecThreads = 256;
constexpr int kRecTokBlock = 8;  // tokens whose prologue is computed together

// PC: one decay per key channel (p.per_channel), a separate instance so that
// the scalar-decay kernel carries none of its work.
template <int DK, int DV, typename T, bool PC>
__global__ void __launch_bounds__(kRecThreads, 2)
recurrent_kernel(RecurrentArgs p) {
    constexpr int L = DV / 4;            // lanes per state row
    constexpr int RG = kRecThreads / L;  // row groups
    constexpr int RPT = DK / RG;         // rows per thread
    constexpr int CH = 2 * DK + DV;      // channels this head reads: q | k | v
    constexpr int NW = kRecThreads / 32;
    static_assert(DK % RG == 0 && RPT >= 1, "unsupported head dims");

    __shared__ float cbuf[kRecTokBlock][CH];
    __shared__ float gam[kRecTokBlock], bet[kRecTokBlock], kqs[kRecTokBlock];
    __shared__ float gamc[PC ? kRecTokBlock : 1][PC ? DK : 1];  // per key channel
    __shared__ float red[NW][2][DV];
    __shared__ __align__(16) float dlt[DV];  // read back as float4
    __shared__ float ysum[DV / 32];

    const int hv = blockIdx.x;
    const int n = blockIdx.y;
    const int hv_n = p.n_v_heads;
    const int hk = key_head(hv, hv_n / p.n_k_heads, p.n_k_heads, p.head_map);
    const int cd = 2 * p.n_k_heads * DK + hv_n * DV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = tid % L, rg = tid / L;
    const int K = p.conv_k, keep = K - 1;

    int bos, len;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - bos;
    } else {
        bos = n * p.uniform_T;
        len = p.uniform_T;
    }

    const T* __restrict__ x = static_cast<const T*>(p.x);
    const T* __restrict__ z = static_cast<const T*>(p.z);
    const T* __restrict__ av = static_cast<const T*>(p.a);
    const T* __restrict__ bv = static_cast<const T*>(p.b);
    const T* __restrict__ cs_in = static_cast<const T*>(p.conv_state_in);
    T* __restrict__ out = static_cast<T*>(p.out);

    // Issue the state loads first; they stay in flight during the prologue.
    const size_t slab = ((size_t)n * hv_n + hv) * DK * DV;
    float4 s[RPT];
    if (p.state_in) {
        const float4* src = reinterpret_cast<const float4*>(p.state_in + slab);
#pragma unroll
        for (int i = 0; i < RPT; ++i) s[i] = src[(rg + RG * i) * L + c4];
    } else {
#pragma unroll
        for (int i = 0; i < RPT; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    for (int t0 = 0; t0 < len; t0 += kRecTokBlock) {
        const int nb = min(kRecTokBlock, len - t0);
        // ---- prologue: conv + SiLU for nb tokens x (q | k | v) channels
        for (int idx = tid; idx < nb * CH; idx += kRecThreads) {
            const int tau = idx / CH, lc = idx % CH;
            const int ch = lc < DK ? hk * DK + lc
                         : lc < 2 * DK ? p.n_k_heads * DK + hk * DK + (lc - DK)
                                       : 2 * p.n_k_heads * DK + hv * DV + (lc - 2 * DK);
            const int t = bos + t0 + tau;
            float acc = 0.f;
            for (int j = 0; j < K; ++j) {
                const int src = t - keep + j;
                float v;
                if (src >= bos)
                    v = to_f32(x[(size_t)src * cd + ch]);
                else if (cs_in)
                    v = to_f32(cs_in[((size_t)n * cd + ch) * keep + keep + (src - bos)]);
                else
                    v = 0.f;
                acc = fmaf(p.conv_w[(size_t)ch * K + j], v, acc);
            }
            cbuf[tau][lc] = siluf_(acc);
        }
        if (tid < nb) {
            const size_t gi = (size_t)(bos + t0 + tid) * hv_n + hv;
            if (!PC)
                gam[tid] = expf(log_decay(to_f32(av[gi]), p.A_log[hv], p.dt_bias[hv], p.decay_form));
            bet[tid] = sigmoidf_(to_f32(bv[gi]));
        }
        if (PC) {  // S <- diag(e^{g_t}) S: one decay per key channel (state row)
            for (int idx = tid; idx < nb * DK; idx += kRecThreads) {
                const int tau = idx / DK, r = idx % DK;
                const size_t gi = ((size_t)(bos + t0 + tau) * hv_n + hv) * DK + r;
                gamc[tau][r] = expf(log_decay(to_f32(av[gi]), p.A_log[hv], p.dt_bias[(size_t)hv * DK + r],
                                              p.decay_form));
            }
            if (tid < nb) gam[tid] = 1.f;  // the decay sits on the rows instead
        }
        __syncthreads();
        // ---- L2-normalise q and k of each token (one warp per token), k.q
        if (warp < nb) {
            float qs = 0.f, ks = 0.f;
            for (int i = lane; i < DK; i += 32) {
                const float q = cbuf[warp][i], k = cbuf[warp][DK + i];
                qs = fmaf(q, q, qs);
                ks = fmaf(k, k, ks);
            }
            qs = group_sum<32>(qs);
            ks = group_sum<32>(ks);
            const float qi = rsqrtf(qs + p.l2_eps) * rsqrtf((float)DK);
            const float ki = rsqrtf(ks + p.l2_eps);
            float d = 0.f;
            for (int i = lane; i < DK; i += 32) {
                const float q = cbuf[warp][i] * qi, k = cbuf[warp][DK + i] * ki;
                cbuf[warp][i] = q;
                cbuf[warp][DK + i] = k;
                d = fmaf(q, k, d);
            }
            d = group_sum<32>(d);
            if (lane == 0) kqs[warp] = d;
        }
        __syncthreads();

        // ---- the delta rule, token by token
        for (int tau = 0; tau < nb; ++tau) {
            const int t = bos + t0 + tau;
            const float gm = gam[tau], bt = bet[tau], gm_h = gm;
            float kv[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = rg + RG * i;
                // with per-channel decays, S^T k and S^T q of the decayed state
                // fold row r's decay into k_r and q_r
                const float fr = PC ? gamc[tau][r] : 1.f;
                const float kr = cbuf[tau][DK + r] * fr, qr = cbuf[tau][r] * fr;
                kv[0] = fmaf(s[i].x, kr, kv[0]); sq[0] = fmaf(s[i].x, qr, sq[0]);
                kv[1] = fmaf(s[i].y, kr, kv[1]); sq[1] = fmaf(s[i].y, qr, sq[1]);
                kv[2] = fmaf(s[i].z, kr, kv[2]); sq[2] = fmaf(s[i].z, qr, sq[2]);
                kv[3] = fmaf(s[i].w, kr, kv[3]); sq[3] = fmaf(s[i].w, qr, sq[3]);
            }
#pragma unroll
            for (int off = L; off < 32; off <<= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kv[e] += __shfl_xor_sync(0xffffffffu, kv[e], off);
                    sq[e] += __shfl_xor_sync(0xffffffffu, sq[e], off);
                }
            }
            if (lane < L) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    red[warp][0][c4 * 4 + e] = kv[e];
                    red[warp][1][c4 * 4 + e] = sq[e];
                }
            }
            __syncthreads();
            float o = 0.f;
            if (tid < DV) {
                float kvc = 0.f, sqc = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    kvc += red[w][0][tid];
                    sqc += red[w][1][tid];
                }
                const float d = bt * (cbuf[tau][2 * DK + tid] - gm * kvc);
                o = fmaf(kqs[tau], d, gm * sqc);
                dlt[tid] = d;
                const float o2 = group_sum<32>(o * o);
                if (lane == 0) ysum[warp] = o2;
            }
            __syncthreads();
            if (tid < DV) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < DV / 32; ++w) tot += ysum[w];
                const float rr = rsqrtf(tot / (float)DV + p.rms_eps);
                const size_t oi = (size_t)t * hv_n * DV + (size_t)hv * DV + tid;
                const float y = o * rr * p.norm_w[tid] * gatef_(to_f32(z[oi]), p.act);
                out[oi] = from_f32<T>(y);
            }
            const float4 dv4 = *reinterpret_cast<const float4*>(&dlt[c4 * 4]);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float kr = cbuf[tau][DK + rg + RG * i];
                const float gm = PC ? gamc[tau][rg + RG * i] : gm_h;
                s[i].x = fmaf(gm, s[i].x, kr * dv4.x);
                s[i].y = fmaf(gm, s[i].y, kr * dv4.y);
                s[i].z = fmaf(gm, s[i].z, kr * dv4.z);
                s[i].w = fmaf(gm, s[i].w, kr * dv4.w);
            }
            if (p.inter) {
                float4* dst = reinterpret_cast<float4*>(p.inter + ((size_t)t * hv_n + hv) * DK * DV);
#pragma unroll
                for (int i = 0; i < RPT; ++i) dst[(rg + RG * i) * L + c4] = s[i];
            }
        }
        __syncthreads();
    }

    if (p.state_out) {
        float4* dst = reinterpret_cast<float4*>(p.state_out + slab);
#pragma unroll
        for (int i = 0; i < RPT; ++i) dst[(rg + RG * i) * L + c4] = s[i];
    }
}

template <typename T>
static cudaError_t launch_recurrent_t(const RecurrentArgs& p, int dk, int dv, cudaStream_t st) {
    dim3 grid(p.n_v_heads, p.n_seq);
#define GDN_REC_CASE(A, B)                                                        \
    if (dk == A && dv == B) {                                                     \
        if (p.per_channel)                                                        \
            recurrent_kernel<A, B, T, true><<<grid, kRecThreads, 0, st>>>(p);     \
        else                                                                      \
            recurrent_kernel<A, B, T, false><<<grid, kRecThreads, 0, st>>>(p);    \
        return cudaGetLastError();                                                \
    }
    GDN_REC_CASE(32, 32) GDN_REC_CASE(32, 64) GDN_REC_CASE(32, 128)
    GDN_REC_CASE(64, 32) GDN_REC_CASE(64, 64) GDN_REC_CASE(64, 128)
    GDN_REC_CASE(128, 32) GDN_REC_CASE(128, 64) GDN_REC_CASE(128, 128)
#undef GDN_REC_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_recurrent(const RecurrentArgs& p, int dk, int dv, bool bf16, cudaStream_t st) {
    if (p.n_seq == 0) return cudaSuccess;
    return bf16 ? launch_recurrent_t<__nv_bfloat16>(p, dk, dv, st)
                : launch_recurrent_t<float>(p, dk, dv, st);
}

// Keep an accepted prefix of a verify call: state <- inter[n, accepted-1].
__global__ void __launch_bounds__(256) commit_state_kernel(CommitArgs p) {
    const int hv = blockIdx.x, n = blockIdx.y;
    const int j = min(max(p.accepted[n], 0), p.T);
    if (j == 0) return;
    const size_t slab = (size_t)p.d_k * p.d_v;
    const float4* src = reinterpret_cast<const float4*>(
        p.inter + (((size_t)n * p.T + (j - 1)) * p.n_v_heads + hv) * slab);
    float4* dst = reinterpret_cast<float4*>(p.state + ((size_t)n * p.n_v_heads + hv) * slab);
    for (size_t i = threadIdx.x; i < slab / 4; i += blockDim.x) dst[i] = src[i];
}

cudaError_t launch_commit_state(const CommitArgs& p, cudaStream_t st) {
    if (p.n_seq == 0) return cudaSuccess;
    commit_state_kernel<<<dim3(p.n_v_heads, p.n_seq), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
