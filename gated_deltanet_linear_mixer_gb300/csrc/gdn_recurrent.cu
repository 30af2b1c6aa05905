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
#include "gdn_tc.cuh"

namespace gdn {

constexpr int kRecThreads = 256;
constexpr int kRecTokBlock = 8;  // tokens whose prologue is computed together

template <int DK, int DV, typename T>
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
    __shared__ float red[NW][2][DV];
    __shared__ __align__(16) float dlt[DV];  // read back as float4
    __shared__ float ysum[DV / 32];

    const int hv = blockIdx.x;
    const int n = blockIdx.y;
    const int hv_n = p.n_v_heads;
    const int hk = hv / (hv_n / p.n_k_heads);
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
            gam[tid] = expf(log_decay(to_f32(av[gi]), p.A_log[hv], p.dt_bias[hv]));
            bet[tid] = sigmoidf_(to_f32(bv[gi]));
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
            const float gm = gam[tau], bt = bet[tau];
            float kv[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = rg + RG * i;
                const float kr = cbuf[tau][DK + r], qr = cbuf[tau][r];
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
        recurrent_kernel<A, B, T><<<grid, kRecThreads, 0, st>>>(p);               \
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


// ===================================================================== //
// Persistent, pipelined decode.
//
// One CTA per SM (256 threads) walks its share of the (sequence, key head)
// groups and, inside a group, the value heads that share the key head.  For
// each value head the whole working set -- the d_k x d_v fp32 state slab, the
// q | k | v channels of the T tokens, their conv history, the conv weights
// and z -- is brought into one stage of a shared-memory ring by 1-D bulk
// copies (cp.async.bulk) issued n_stages-1 heads ahead, so HBM keeps
// streaming while the current head is computed.  The arithmetic is that of
// recurrent_kernel.  Because a group's value heads run back to back on one
// CTA, the conv history is updated in place here: v channels after each
// head, the shared q/k channels after the group's last head.
// ===================================================================== //

__device__ int g_decode_error = 0;

namespace {

template <typename T>
struct StageLayout {
    uint32_t xq, xk, xv, hq, hk, hv, wq, wk, wv, z, bytes;
    __host__ __device__ StageLayout(int dk, int dv, int tn, int km1, int K) {
        auto up = [](uint32_t v) { return (v + 127u) & ~127u; };
        uint32_t o = static_cast<uint32_t>(dk) * dv * 4;
        xq = o; o = up(o + tn * dk * sizeof(T));
        xk = o; o = up(o + tn * dk * sizeof(T));
        xv = o; o = up(o + tn * dv * sizeof(T));
        hq = o; o = up(o + dk * km1 * sizeof(T));
        hk = o; o = up(o + dk * km1 * sizeof(T));
        hv = o; o = up(o + dv * km1 * sizeof(T));
        wq = o; o = up(o + dk * K * 4);
        wk = o; o = up(o + dk * K * 4);
        wv = o; o = up(o + dv * K * 4);
        z = o; o = up(o + tn * dv * sizeof(T));
        bytes = o;
    }
};

}  // namespace

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kRecThreads, 1)
decode_stream_kernel(DecodeArgs p) {
    constexpr int L = DV / 4, RG = kRecThreads / L, RPT = DK / RG, CH = 2 * DK + DV;
    constexpr int NW = kRecThreads / 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                               ~static_cast<uintptr_t>(127));
    __shared__ __align__(8) uint64_t bars[3];
    __shared__ float gam[16], bet[16], kqs[16];
    __shared__ float red[NW][2][DV];
    __shared__ __align__(16) float dlt[DV];  // read back as float4
    __shared__ float ysum[DV / 32];
    __shared__ float s_norm_w[DV];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = tid % L, rg = tid / L;
    const int Tn = p.T, K = p.conv_k, km1 = K - 1;
    const int hk_n = p.n_k_heads, hv_n = p.n_v_heads, R = hv_n / hk_n;
    const int cd = 2 * hk_n * DK + hv_n * DV;
    const int n_groups = p.n_seq * hk_n;
    const int G = gridDim.x;
    const int my_groups = blockIdx.x < n_groups ? (n_groups - 1 - blockIdx.x) / G + 1 : 0;
    const int n_items = my_groups * R;
    const int S = p.n_stages;
    const StageLayout<T> lay(DK, DV, Tn, km1, K);
    float* cbuf = reinterpret_cast<float*>(smem + S * p.stage_bytes);  // [Tn][CH]

    const T* __restrict__ x = static_cast<const T*>(p.x);
    const T* __restrict__ z = static_cast<const T*>(p.z);
    const T* __restrict__ av = static_cast<const T*>(p.a);
    const T* __restrict__ bv = static_cast<const T*>(p.b);
    T* __restrict__ cs = static_cast<T*>(p.conv_state);
    T* __restrict__ out = static_cast<T*>(p.out);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) tc::mbar_init(&bars[i], 1);
        tc::fence_barrier_init();
    }
    for (int i = tid; i < DV; i += kRecThreads) s_norm_w[i] = p.norm_w[i];
    __syncthreads();

    // Item -> (sequence, key head, value head).
    auto item_pos = [&](int item, int& n, int& hk, int& hv, int& r) {
        const int g = blockIdx.x + (item / R) * G;
        r = item % R;
        n = g / hk_n;
        hk = g % hk_n;
        hv = hk * R + r;
    };
    // Warp 0 brings item `item`'s working set into its stage.
    auto issue = [&](int item) {
        int n, hk, hv, r;
        item_pos(item, n, hk, hv, r);
        const int s = item % S;
        uint8_t* st = smem + s * p.stage_bytes;
        const int n_copies = 1 + 4 * Tn + 3 + (cs ? 3 : 0);
        const uint32_t bytes = DK * DV * 4 + sizeof(T) * (Tn * (2 * DK + DV) + Tn * DV) +
                               4u * K * (2 * DK + DV) + (cs ? sizeof(T) * km1 * (2 * DK + DV) : 0u);
        if (lane == 0) tc::mbar_arrive_expect_tx(&bars[s], bytes);
        __syncwarp();
        for (int k = lane; k < n_copies; k += 32) {
            if (k == 0) {
                tc::bulk_load(st, p.state + ((size_t)n * hv_n + hv) * DK * DV, DK * DV * 4, &bars[s]);
            } else if (k <= 3 * Tn) {
                const int t = (k - 1) / 3, part = (k - 1) % 3;
                const size_t row = ((size_t)n * Tn + t) * cd;
                if (part == 0)
                    tc::bulk_load(st + lay.xq + t * DK * sizeof(T), x + row + hk * DK, DK * sizeof(T), &bars[s]);
                else if (part == 1)
                    tc::bulk_load(st + lay.xk + t * DK * sizeof(T), x + row + hk_n * DK + hk * DK,
                                  DK * sizeof(T), &bars[s]);
                else
                    tc::bulk_load(st + lay.xv + t * DV * sizeof(T), x + row + 2 * hk_n * DK + hv * DV,
                                  DV * sizeof(T), &bars[s]);
            } else if (k <= 4 * Tn) {
                const int t = k - 1 - 3 * Tn;
                tc::bulk_load(st + lay.z + t * DV * sizeof(T),
                              z + ((size_t)n * Tn + t) * hv_n * DV + hv * DV, DV * sizeof(T), &bars[s]);
            } else if (k <= 4 * Tn + 3) {
                const int part = k - 1 - 4 * Tn;
                const int ch0 = part == 0 ? hk * DK : part == 1 ? hk_n * DK + hk * DK
                                                                : 2 * hk_n * DK + hv * DV;
                const int nch = part == 2 ? DV : DK;
                tc::bulk_load(st + (part == 0 ? lay.wq : part == 1 ? lay.wk : lay.wv),
                              p.conv_w + (size_t)ch0 * K, nch * K * 4, &bars[s]);
            } else {
                const int part = k - 2 - 4 * Tn - 3 + 1;
                const int ch0 = part == 0 ? hk * DK : part == 1 ? hk_n * DK + hk * DK
                                                                : 2 * hk_n * DK + hv * DV;
                const int nch = part == 2 ? DV : DK;
                tc::bulk_load(st + (part == 0 ? lay.hq : part == 1 ? lay.hk : lay.hv),
                              cs + ((size_t)n * cd + ch0) * km1, nch * km1 * sizeof(T), &bars[s]);
            }
        }
    };

    const int prologue_items = n_items < S ? n_items : S;
    if (warp == 0)
        for (int i = 0; i < prologue_items; ++i) issue(i);
    // gate inputs of item 0 (scalars; loaded one item ahead into registers)
    float a_nx = 0.f, b_nx = 0.f, alog_nx = 0.f, dtb_nx = 0.f;
    auto load_gates = [&](int item) {
        if (item < n_items && tid < Tn) {
            int n, hk, hv, r;
            item_pos(item, n, hk, hv, r);
            const size_t gi = ((size_t)n * Tn + tid) * hv_n + hv;
            a_nx = to_f32(av[gi]);
            b_nx = to_f32(bv[gi]);
            alog_nx = p.A_log[hv];
            dtb_nx = p.dt_bias[hv];
        }
    };
    load_gates(0);

    int consumed = 0;
    bool dead = false;
    for (int i = 0; i < n_items; ++i) {
        int n, hk, hv, r;
        item_pos(i, n, hk, hv, r);
        const int s = i % S;
        const uint8_t* st = smem + s * p.stage_bytes;
        const float a_cur = a_nx, b_cur = b_nx, alog_cur = alog_nx, dtb_cur = dtb_nx;
        load_gates(i + 1);
        if (__syncthreads_or(tc::mbar_wait(&bars[s], (i / S) & 1) ? 0 : 1)) {
            if (tid == 0) atomicCAS(&g_decode_error, 0, 1);
            dead = true;
            break;
        }
        consumed = i + 1;
        // ---- prologue: conv + SiLU for Tn tokens x (q | k | v) channels
        const T* sxq = reinterpret_cast<const T*>(st + lay.xq);
        const T* sxk = reinterpret_cast<const T*>(st + lay.xk);
        const T* sxv = reinterpret_cast<const T*>(st + lay.xv);
        const T* shq = reinterpret_cast<const T*>(st + lay.hq);
        const T* shk = reinterpret_cast<const T*>(st + lay.hk);
        const T* shv = reinterpret_cast<const T*>(st + lay.hv);
        for (int idx = tid; idx < Tn * CH; idx += kRecThreads) {
            const int tau = idx / CH, lc = idx % CH;
            const T* xs;
            const T* hs;
            const float* ws;
            int c, w;
            if (lc < DK) { xs = sxq; hs = shq; ws = reinterpret_cast<const float*>(st + lay.wq); c = lc; w = DK; }
            else if (lc < 2 * DK) { xs = sxk; hs = shk; ws = reinterpret_cast<const float*>(st + lay.wk); c = lc - DK; w = DK; }
            else { xs = sxv; hs = shv; ws = reinterpret_cast<const float*>(st + lay.wv); c = lc - 2 * DK; w = DV; }
            float acc = 0.f;
            for (int j = 0; j < K; ++j) {
                const int src = tau - km1 + j;
                float v;
                if (src >= 0) v = to_f32(xs[src * w + c]);
                else if (cs) v = to_f32(hs[c * km1 + km1 + src]);
                else v = 0.f;
                acc = fmaf(ws[c * K + j], v, acc);
            }
            cbuf[tau * CH + lc] = siluf_(acc);
        }
        if (tid < Tn) {
            gam[tid] = expf(log_decay(a_cur, alog_cur, dtb_cur));
            bet[tid] = sigmoidf_(b_cur);
        }
        __syncthreads();
        for (int tau = warp; tau < Tn; tau += NW) {  // L2 norms of q, k and k.q
            float* cb = cbuf + tau * CH;
            float qs = 0.f, ks = 0.f;
            for (int e = lane; e < DK; e += 32) {
                qs = fmaf(cb[e], cb[e], qs);
                ks = fmaf(cb[DK + e], cb[DK + e], ks);
            }
            qs = group_sum<32>(qs);
            ks = group_sum<32>(ks);
            const float qi = rsqrtf(qs + p.l2_eps) * rsqrtf((float)DK);
            const float ki = rsqrtf(ks + p.l2_eps);
            float d = 0.f;
            for (int e = lane; e < DK; e += 32) {
                const float q = cb[e] * qi, k = cb[DK + e] * ki;
                cb[e] = q;
                cb[DK + e] = k;
                d = fmaf(q, k, d);
            }
            d = group_sum<32>(d);
            if (lane == 0) kqs[tau] = d;
        }
        // state slab from the stage into registers
        float4 sreg[RPT];
        {
            const float4* sst = reinterpret_cast<const float4*>(st);
#pragma unroll
            for (int k = 0; k < RPT; ++k) sreg[k] = sst[(rg + RG * k) * L + c4];
        }
        __syncthreads();
        const T* sz = reinterpret_cast<const T*>(st + lay.z);
        for (int tau = 0; tau < Tn; ++tau) {
            const float* cb = cbuf + tau * CH;
            const float gm = gam[tau], bt = bet[tau];
            float kv[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                const int row = rg + RG * k;
                const float kr = cb[DK + row], qr = cb[row];
                kv[0] = fmaf(sreg[k].x, kr, kv[0]); sq[0] = fmaf(sreg[k].x, qr, sq[0]);
                kv[1] = fmaf(sreg[k].y, kr, kv[1]); sq[1] = fmaf(sreg[k].y, qr, sq[1]);
                kv[2] = fmaf(sreg[k].z, kr, kv[2]); sq[2] = fmaf(sreg[k].z, qr, sq[2]);
                kv[3] = fmaf(sreg[k].w, kr, kv[3]); sq[3] = fmaf(sreg[k].w, qr, sq[3]);
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
                const float d = bt * (cb[2 * DK + tid] - gm * kvc);
                o = fmaf(kqs[tau], d, gm * sqc);
                dlt[tid] = d;
                const float o2 = group_sum<32>(o * o);
                if (lane == 0) ysum[warp] = o2;
            }
            __syncthreads();
            const size_t tok = (size_t)n * Tn + tau;
            if (tid < DV) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < DV / 32; ++w) tot += ysum[w];
                const float rr = rsqrtf(tot / (float)DV + p.rms_eps);
                const float y = o * rr * s_norm_w[tid] * gatef_(to_f32(sz[tau * DV + tid]), p.act);
                out[tok * hv_n * DV + (size_t)hv * DV + tid] = from_f32<T>(y);
            }
            const float4 dv4 = *reinterpret_cast<const float4*>(&dlt[c4 * 4]);
#pragma unroll
            for (int k = 0; k < RPT; ++k) {
                const float kr = cb[DK + rg + RG * k];
                sreg[k].x = fmaf(gm, sreg[k].x, kr * dv4.x);
                sreg[k].y = fmaf(gm, sreg[k].y, kr * dv4.y);
                sreg[k].z = fmaf(gm, sreg[k].z, kr * dv4.z);
                sreg[k].w = fmaf(gm, sreg[k].w, kr * dv4.w);
            }
            if (p.inter) {
                float4* dst = reinterpret_cast<float4*>(p.inter + (tok * hv_n + hv) * DK * DV);
#pragma unroll
                for (int k = 0; k < RPT; ++k) dst[(rg + RG * k) * L + c4] = sreg[k];
            }
        }
        if (!p.inter) {
            float4* dst = reinterpret_cast<float4*>(p.state + ((size_t)n * hv_n + hv) * DK * DV);
#pragma unroll
            for (int k = 0; k < RPT; ++k) dst[(rg + RG * k) * L + c4] = sreg[k];
        }
        if (p.write_conv && cs) {
            // new history = last K-1 raw inputs, oldest first: v channels of this
            // head; q and k channels once the group's last head is done
            const int nch = DV + (r == R - 1 ? 2 * DK : 0);
            for (int idx = tid; idx < nch * km1; idx += kRecThreads) {
                const int e = idx / km1, slot = idx % km1;
                const T* xs;
                const T* hs;
                int c, w, ch0;
                if (e < DV) { xs = sxv; hs = shv; c = e; w = DV; ch0 = 2 * hk_n * DK + hv * DV; }
                else if (e < DV + DK) { xs = sxq; hs = shq; c = e - DV; w = DK; ch0 = hk * DK; }
                else { xs = sxk; hs = shk; c = e - DV - DK; w = DK; ch0 = hk_n * DK + hk * DK; }
                const int ti = Tn - km1 + slot;
                const T v = ti >= 0 ? xs[ti * w + c] : hs[c * km1 + km1 + ti];
                cs[((size_t)n * cd + ch0 + c) * km1 + slot] = v;
            }
        }
        __syncthreads();  // stage s and cbuf are free again
        if (warp == 0 && i + S < n_items) issue(i + S);
    }
    if (dead) {  // let copies already in flight land before the CTA exits
        const int issued = n_items < consumed + S ? n_items : consumed + S;
        for (int i = consumed; i < issued; ++i) tc::mbar_wait(&bars[i % S], (i / S) & 1);
    }
}

template <typename T>
static cudaError_t launch_decode_stream_t(DecodeArgs p, int dk, int dv, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const StageLayout<T> lay(dk, dv, p.T, p.conv_k - 1, p.conv_k);
    p.stage_bytes = lay.bytes;
    const size_t cbuf = (size_t)p.T * (2 * dk + dv) * 4;
    p.n_stages = 3 * (size_t)lay.bytes + cbuf + 128 <= 200 * 1024 ? 3 : 2;
    const size_t smem = (size_t)p.n_stages * lay.bytes + cbuf + 128;
    const int groups = p.n_seq * p.n_k_heads;
    const int grid = groups < sms ? groups : sms;
#define GDN_DEC_CASE(A, B)                                                                   \
    if (dk == A && dv == B) {                                                                \
        e = cudaFuncSetAttribute(decode_stream_kernel<A, B, T>,                              \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);    \
        if (e != cudaSuccess) return e;                                                      \
        decode_stream_kernel<A, B, T><<<grid, kRecThreads, smem, st>>>(p);                   \
        return cudaGetLastError();                                                           \
    }
    GDN_DEC_CASE(32, 32) GDN_DEC_CASE(32, 64) GDN_DEC_CASE(32, 128)
    GDN_DEC_CASE(64, 32) GDN_DEC_CASE(64, 64) GDN_DEC_CASE(64, 128)
    GDN_DEC_CASE(128, 32) GDN_DEC_CASE(128, 64) GDN_DEC_CASE(128, 128)
#undef GDN_DEC_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_stream(DecodeArgs p, int dk, int dv, bool bf16, cudaStream_t st) {
    if (p.n_seq == 0) return cudaSuccess;
    return bf16 ? launch_decode_stream_t<__nv_bfloat16>(p, dk, dv, st)
                : launch_decode_stream_t<float>(p, dk, dv, st);
}

cudaError_t read_decode_error(int* code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_decode_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int));
    }
    return e;
}

}  // namespace gdn
