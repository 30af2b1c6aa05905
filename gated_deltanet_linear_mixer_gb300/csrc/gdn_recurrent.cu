// Token-recurrent GDN kernel: the decode path (one or a few tokens per
// sequence against a resident fp32 state) and the fp32 prefill path.
//
// It runs the delta rule exactly as cherenkov qwen4_exp/cpu.rs fn deltanet
// and oxinfer 0.0.5 src/qwen.rs DeltaRule::run define it (decay, read of the
// decayed state, rank-one write, readout), with the conv/normalise/gate
// prologue and the gated-RMSNorm epilogue fused in.
//
// Design (memory-bound): persistent CTAs of 256 threads, two per SM, each
// walking (sequence, value head) items.  The d_k x d_v fp32 state slab of an
// item is streamed from HBM once, held in registers for all the tokens of the
// call, and written back once; while an item computes, the next item's slab
// is already on its way into shared memory (one bulk async copy), so every
// SM keeps two slabs of loads in flight between its items.  The inputs of an
// item's first token block (its q|k|v rows, conv history and weights, z rows)
// come into shared memory by per-thread async copies issued together with the
// gate loads at the start of the item, so that they cost one round trip to
// memory instead of one per dependent load.  Thread layout: a
// state row (d_v floats) is covered by d_v/4 lanes with one float4 each, so
// every load/store instruction of a warp moves whole 128..512-byte rows; the
// CTA's row groups split the d_k rows.  The two per-token column reductions
// S^T k and S^T q share one pass: warp shuffles across the row groups inside
// a warp, then shared memory across warps.  The readout uses
// o = e^g S^T q + (k.q) delta, which equals S'^T q for the written state S'
// (S' = e^g S + k delta^T), so the state is read once per token.
//
// A second kernel, verify_ro_kernel, takes verify calls that write no state:
// all of a sequence's drafts in one pass over the state (the rule unrolled
// over up to four tokens), with no state update.
#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

constexpr int kRecThreads = 256;
constexpr int kRecTokBlock = 8;  // tokens whose prologue is computed together
constexpr int kRecCtasPerSm = 2;

// This file's device error word: 30 = a CTA's wait for its state copy gave up.
__device__ int g_rec_error = 0;

// 16-byte asynchronous copy global -> shared (cp.async, tracked per thread).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Dynamic shared-memory layout of recurrent_kernel (byte offsets; every
// region 16-byte aligned).
template <int DK, int DV, typename T> struct RecStage {
    static constexpr int CH = 2 * DK + DV;
    static constexpr uint32_t kX = DK * DV * 4;
    static constexpr uint32_t kCs = kX + kRecTokBlock * CH * sizeof(T);
    static constexpr uint32_t kW = kCs + ((CH * 3 * sizeof(T) + 15) / 16) * 16;
    static constexpr uint32_t kZ = kW + CH * 4 * 4;
    static constexpr uint32_t kBytes = kZ + kRecTokBlock * DV * sizeof(T);
};

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
    // A conv-history update launched after this kernel as its programmatic
    // dependent may start on SMs this grid leaves free: it only reads what this
    // kernel reads before waiting for the grid's completion to store.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    __shared__ float cbuf[kRecTokBlock][CH];
    __shared__ float gam[kRecTokBlock], bet[kRecTokBlock], kqs[kRecTokBlock];
    __shared__ float gamc[PC ? kRecTokBlock : 1][PC ? DK : 1];  // per key channel
    __shared__ float red[NW][2][DV];
    __shared__ __align__(16) float dlt[DV];  // read back as float4
    __shared__ float ysum[DV / 32];
    __shared__ __align__(8) uint64_t bar_s;  // the state copy of the CTA's next item
    // dynamic shared memory: that copy [DK][DV], then the raw inputs of an
    // item's first token block (async copies): q | k | v rows, conv history
    // [channel][K-1], conv weights [channel][K], z rows
    extern __shared__ __align__(128) float s_next[];
    using Stage = RecStage<DK, DV, T>;
    uint8_t* dyn = reinterpret_cast<uint8_t*>(s_next);
    T (*st_x)[CH] = reinterpret_cast<T (*)[CH]>(dyn + Stage::kX);
    T* st_cs = reinterpret_cast<T*>(dyn + Stage::kCs);
    float* st_w = reinterpret_cast<float*>(dyn + Stage::kW);
    T (*st_z)[DV] = reinterpret_cast<T (*)[DV]>(dyn + Stage::kZ);

    const int hv_n = p.n_v_heads;
    const int cd = 2 * p.n_k_heads * DK + hv_n * DV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = tid % L, rg = tid / L;
    const int K = p.conv_k, keep = K - 1;
    const int n_items = p.n_seq * hv_n;  // item = n * Hv + hv: also its state slab's index
    constexpr uint32_t kSlabBytes = DK * DV * 4;

    if (tid == 0) {
        tc::mbar_init(&bar_s, 1);
        tc::fence_barrier_init();
    }
    __syncthreads();
    auto issue_state = [&](int item) {  // one thread: the slab in 16 KB pieces
        tc::mbar_arrive_expect_tx(&bar_s, kSlabBytes);
        for (uint32_t off = 0; off < kSlabBytes; off += 16384)
            tc::bulk_load_1d(reinterpret_cast<uint8_t*>(s_next) + off,
                             p.state_in + (size_t)item * DK * DV + off / 4, min(16384u, kSlabBytes - off),
                             &bar_s);
    };
    uint32_t s_phase = 0;
    bool s_pending = p.state_in && (int)blockIdx.x < n_items;
    if (s_pending && tid == 0) issue_state(blockIdx.x);

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int n = item / hv_n, hv = item - n * hv_n;
    const int hk = key_head(hv, hv_n / p.n_k_heads, p.n_k_heads, p.head_map);

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

    // Async copies of the first token block's inputs (every range is a
    // multiple of 16 bytes at a 16-byte aligned offset of its array, given
    // 16-byte aligned bases, which `staged` checks), and its gate inputs.
    const int nb0 = min(kRecTokBlock, len);
    const bool staged = len > 0 && ((reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.z) |
                                     reinterpret_cast<uintptr_t>(p.conv_w) |
                                     reinterpret_cast<uintptr_t>(cs_in)) & 15) == 0;
    float a_pre = 0.f, b_pre = 0.f;
    if (staged) {
        constexpr int QC = DK * (int)sizeof(T) / 16, XC = CH * (int)sizeof(T) / 16;
        const int chq = hk * DK, chk = p.n_k_heads * DK + hk * DK, chv = 2 * p.n_k_heads * DK + hv * DV;
        // chunk c of a q|k|v list with per_q chunks per key range: first channel, chunk within
        auto range_of = [&](int c, int per_q, int& ch, int& off) {
            const int r = c < per_q ? 0 : c < 2 * per_q ? 1 : 2;
            ch = r == 0 ? chq : r == 1 ? chk : chv;
            off = c - r * per_q;
        };
        for (int i = tid; i < nb0 * XC; i += kRecThreads) {
            const int tau = i / XC, c = i - tau * XC;
            int ch, off;
            range_of(c, QC, ch, off);
            cp_async16(reinterpret_cast<uint4*>(&st_x[tau][0]) + c,
                       reinterpret_cast<const uint4*>(x + (size_t)(bos + tau) * cd + ch) + off);
        }
        if (cs_in) {
            const int per_q = QC * keep, tot = (2 * DK + DV) * (int)sizeof(T) * keep / 16;
            for (int c = tid; c < tot; c += kRecThreads) {
                int ch, off;
                range_of(c, per_q, ch, off);
                cp_async16(reinterpret_cast<uint4*>(st_cs) + c,
                           reinterpret_cast<const uint4*>(cs_in + ((size_t)n * cd + ch) * keep) + off);
            }
        }
        {
            const int per_q = DK * K / 4, tot = CH * K / 4;
            for (int c = tid; c < tot; c += kRecThreads) {
                int ch, off;
                range_of(c, per_q, ch, off);
                cp_async16(reinterpret_cast<uint4*>(st_w) + c,
                           reinterpret_cast<const uint4*>(p.conv_w + (size_t)ch * K) + off);
            }
        }
        constexpr int ZC = DV * (int)sizeof(T) / 16;
        for (int i = tid; i < nb0 * ZC; i += kRecThreads) {
            const int tau = i / ZC, c = i - tau * ZC;
            cp_async16(reinterpret_cast<uint4*>(&st_z[tau][0]) + c,
                       reinterpret_cast<const uint4*>(z + ((size_t)(bos + tau) * hv_n + hv) * DV) + c);
        }
        cp_async_commit();
        if (tid < nb0) {
            const size_t gi = (size_t)(bos + tid) * hv_n + hv;
            if (!PC) a_pre = to_f32(av[gi]);
            b_pre = to_f32(bv[gi]);
        }
    }

    // The state: from the copy that was in flight since the previous item;
    // once every thread has taken its rows, the next item's copy is issued.
    const size_t slab = (size_t)item * DK * DV;
    float4 s[RPT];
    if (p.state_in) {
        if (!__syncthreads_and(tc::mbar_wait(&bar_s, s_phase))) {
            if (tid == 0) atomicCAS(&g_rec_error, 0, 30);
            break;
        }
        s_phase ^= 1;
        s_pending = false;
        const float4* src = reinterpret_cast<const float4*>(s_next);
#pragma unroll
        for (int i = 0; i < RPT; ++i) s[i] = src[(rg + RG * i) * L + c4];
        __syncthreads();
        if (item + (int)gridDim.x < n_items) {
            if (tid == 0) issue_state(item + gridDim.x);
            s_pending = true;
        }
    } else {
#pragma unroll
        for (int i = 0; i < RPT; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    for (int t0 = 0; t0 < len; t0 += kRecTokBlock) {
        const int nb = min(kRecTokBlock, len - t0);
        const bool from_stage = staged && t0 == 0;
        // ---- prologue: conv + SiLU for nb tokens x (q | k | v) channels
        if (from_stage) {
            cp_async_wait_all();
            __syncthreads();
            for (int idx = tid; idx < nb * CH; idx += kRecThreads) {
                const int tau = idx / CH, lc = idx % CH;
                float acc = 0.f;
                for (int j = 0; j < K; ++j) {
                    const int tt = tau - keep + j;  // token of the item (this block starts it)
                    const float v = tt >= 0 ? to_f32(st_x[tt][lc])
                                    : cs_in ? to_f32(st_cs[lc * keep + keep + tt]) : 0.f;
                    acc = fmaf(st_w[lc * K + j], v, acc);
                }
                cbuf[tau][lc] = siluf_(acc);
            }
        } else
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
                gam[tid] = expf(log_decay(from_stage ? a_pre : to_f32(av[gi]), p.A_log[hv], p.dt_bias[hv],
                                          p.decay_form));
            bet[tid] = sigmoidf_(from_stage ? b_pre : to_f32(bv[gi]));
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
                const float zv = from_stage ? to_f32(st_z[tau][tid]) : to_f32(z[oi]);
                const float y = o * rr * p.norm_w[tid] * gatef_(zv, p.act);
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
    }  // items

    // no copy may be in flight when the CTA leaves (only after a give-up)
    if (s_pending && tid == 0 && !tc::mbar_wait(&bar_s, s_phase)) atomicCAS(&g_rec_error, 0, 30);
}

// ------------------------------------------------------------ read-only verify
// A verify call that keeps no state (no state_out, no intermediates; at most
// kRecSub tokens per sequence, scalar decay) needs the state only to read it.
// Its tokens then share one pass over the state: with S the state before the
// first token, G_j the decay through token j and D_ij the decay over the
// tokens after i through j,
//   kv_j = G_j S^T k_j + sum_{i<j} D_ij (k_i.k_j) delta_i,
//   delta_j = beta_j (v_j - kv_j),
//   o_j = G_j S^T q_j + sum_{i<=j} D_ij (k_i.q_j) delta_i,
// which is the token-by-token rule (S_j = e^{g_j} S_{j-1} + k_j delta_j^T,
// o_j = S_j^T q_j) unrolled over the call's tokens.  The state is never
// written, so no thread updates it.
constexpr int kRecSub = 4;  // tokens per sequence the read-only kernel takes

// Dynamic shared memory of verify_ro_kernel (byte offsets, 16-byte aligned):
// the next item's state slab; the item's input staging (q|k|v rows, conv
// history, conv weights), reused for the per-warp column sums once the conv
// has read it; the z rows.
template <int DK, int DV, typename T> struct RoStage {
    static constexpr int CH = 2 * DK + DV;
    static constexpr uint32_t kX = DK * DV * 4;
    static constexpr uint32_t kCs = kX + kRecSub * CH * sizeof(T);
    static constexpr uint32_t kW = kCs + ((CH * 3 * sizeof(T) + 15) / 16) * 16;
    static constexpr uint32_t kStageEnd = kW + CH * 4 * 4;
    static constexpr uint32_t kRedEnd = kX + (kRecThreads / 32) * kRecSub * DV * 2 * 4;
    static constexpr uint32_t kZ = kStageEnd > kRedEnd ? kStageEnd : kRedEnd;
    static constexpr uint32_t kBytes = kZ + kRecSub * DV * sizeof(T);
};

// N consecutive floats of a shared-memory row (16-byte vectors when N is a
// multiple of 4, the caller's offset then being one too).
template <int N>
__device__ __forceinline__ void ro_rows(float (&v)[N], const float* src) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 f = *reinterpret_cast<const float4*>(src + i);
            v[i] = f.x;
            v[i + 1] = f.y;
            v[i + 2] = f.z;
            v[i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = src[i];
    }
}

// The one pass over this thread's state rows: S^T k_j and S^T q_j (raw conv
// outputs) for the M tokens, reduced over the warp's row groups and stored
// per warp, key and query sums of a column side by side:
// red[((warp * kRecSub + j) * DV + column) * 2 + {0: key, 1: query}].
template <int M, int DK, int DV, int RPT, int L, int CH>
__device__ __forceinline__ void ro_colsums(const float4 (&s)[RPT], const float (*cbuf)[CH], int rg, int lane,
                                           int warp, int c4, float* red) {
    constexpr int G = RPT % 4 == 0 ? 4 : 1;  // rows per shared-memory load
    float acc[M][2][4];
#pragma unroll
    for (int j = 0; j < M; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][0][e] = acc[j][1][e] = 0.f;
#pragma unroll
    for (int i0 = 0; i0 < RPT; i0 += G) {
#pragma unroll
        for (int j = 0; j < M; ++j) {
            float kr[G], qr[G];
            ro_rows<G>(kr, &cbuf[j][DK + RPT * rg + i0]);
            ro_rows<G>(qr, &cbuf[j][RPT * rg + i0]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 sv = s[i0 + g];
                acc[j][0][0] = fmaf(sv.x, kr[g], acc[j][0][0]);
                acc[j][1][0] = fmaf(sv.x, qr[g], acc[j][1][0]);
                acc[j][0][1] = fmaf(sv.y, kr[g], acc[j][0][1]);
                acc[j][1][1] = fmaf(sv.y, qr[g], acc[j][1][1]);
                acc[j][0][2] = fmaf(sv.z, kr[g], acc[j][0][2]);
                acc[j][1][2] = fmaf(sv.z, qr[g], acc[j][1][2]);
                acc[j][0][3] = fmaf(sv.w, kr[g], acc[j][0][3]);
                acc[j][1][3] = fmaf(sv.w, qr[g], acc[j][1][3]);
            }
        }
    }
#pragma unroll
    for (int off = L; off < 32; off <<= 1)
#pragma unroll
        for (int j = 0; j < M; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[j][0][e] += __shfl_xor_sync(0xffffffffu, acc[j][0][e], off);
                acc[j][1][e] += __shfl_xor_sync(0xffffffffu, acc[j][1][e], off);
            }
    if (lane < L) {
#pragma unroll
        for (int j = 0; j < M; ++j) {
            float4* dst = reinterpret_cast<float4*>(&red[((warp * kRecSub + j) * DV + c4 * 4) * 2]);
            dst[0] = make_float4(acc[j][0][0], acc[j][1][0], acc[j][0][1], acc[j][1][1]);
            dst[1] = make_float4(acc[j][0][2], acc[j][1][2], acc[j][0][3], acc[j][1][3]);
        }
    }
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kRecThreads, 2)
verify_ro_kernel(RecurrentArgs p) {
    constexpr int L = DV / 4;            // lanes per state row
    constexpr int RG = kRecThreads / L;  // row groups
    constexpr int RPT = DK / RG;         // rows per thread (consecutive)
    constexpr int CH = 2 * DK + DV;      // channels this head reads: q | k | v
    constexpr int NW = kRecThreads / 32;
    static_assert(DK % RG == 0 && RPT >= 1 && 2 * DV <= kRecThreads, "unsupported head dims");

    __shared__ __align__(16) float cbuf[kRecSub][CH];  // conv outputs q | k | v (raw)
    __shared__ float gam[kRecSub], bet[kRecSub];
    // the inverse norms of q and k, the decay from the first token through
    // this one, and the normalised, decayed key.key and key.query products with
    // the earlier tokens (the last cfq entry: with the token's own key)
    __shared__ float nq[kRecSub], nk[kRecSub], gcum[kRecSub];
    __shared__ float cfk[kRecSub][kRecSub], cfq[kRecSub][kRecSub];
    __shared__ float ysum[kRecSub][NW];
    __shared__ __align__(8) uint64_t bar_s;  // the state copy of the CTA's next item
    extern __shared__ __align__(128) float s_next[];
    using Stage = RoStage<DK, DV, T>;
    uint8_t* dyn = reinterpret_cast<uint8_t*>(s_next);
    T (*st_x)[CH] = reinterpret_cast<T (*)[CH]>(dyn + Stage::kX);
    T* st_cs = reinterpret_cast<T*>(dyn + Stage::kCs);
    float* st_w = reinterpret_cast<float*>(dyn + Stage::kW);
    float* red = reinterpret_cast<float*>(dyn + Stage::kX);  // after the conv: the column sums
    T (*st_z)[DV] = reinterpret_cast<T (*)[DV]>(dyn + Stage::kZ);

    const int hv_n = p.n_v_heads, m = p.uniform_T;
    const int cd = 2 * p.n_k_heads * DK + hv_n * DV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c4 = tid % L, rg = tid / L;
    const int K = p.conv_k, keep = K - 1;
    const int n_items = p.n_seq * hv_n;
    constexpr uint32_t kSlabBytes = DK * DV * 4;

    if (tid == 0) {
        tc::mbar_init(&bar_s, 1);
        tc::fence_barrier_init();
    }
    __syncthreads();
    auto issue_state = [&](int item) {  // one thread: the slab in 16 KB pieces
        tc::mbar_arrive_expect_tx(&bar_s, kSlabBytes);
        for (uint32_t off = 0; off < kSlabBytes; off += 16384)
            tc::bulk_load_1d(reinterpret_cast<uint8_t*>(s_next) + off,
                             p.state_in + (size_t)item * DK * DV + off / 4, min(16384u, kSlabBytes - off),
                             &bar_s);
    };
    uint32_t s_phase = 0;
    bool s_pending = (int)blockIdx.x < n_items;
    if (s_pending && tid == 0) issue_state(blockIdx.x);

    const T* __restrict__ x = static_cast<const T*>(p.x);
    const T* __restrict__ z = static_cast<const T*>(p.z);
    const T* __restrict__ av = static_cast<const T*>(p.a);
    const T* __restrict__ bv = static_cast<const T*>(p.b);
    const T* __restrict__ cs_in = static_cast<const T*>(p.conv_state_in);
    T* __restrict__ out = static_cast<T*>(p.out);

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int n = item / hv_n, hv = item - n * hv_n;
        const int hk = key_head(hv, hv_n / p.n_k_heads, p.n_k_heads, p.head_map);
        const int bos = n * m;

        // the item's inputs by per-thread async copies (16-byte aligned bases,
        // checked by the host), and its gate inputs
        {
            constexpr int QC = DK * (int)sizeof(T) / 16, XC = CH * (int)sizeof(T) / 16;
            const int chq = hk * DK, chk = p.n_k_heads * DK + hk * DK, chv = 2 * p.n_k_heads * DK + hv * DV;
            auto range_of = [&](int c, int per_q, int& ch, int& off) {
                const int r = c < per_q ? 0 : c < 2 * per_q ? 1 : 2;
                ch = r == 0 ? chq : r == 1 ? chk : chv;
                off = c - r * per_q;
            };
            for (int i = tid; i < m * XC; i += kRecThreads) {
                const int tau = i / XC, c = i - tau * XC;
                int ch, off;
                range_of(c, QC, ch, off);
                cp_async16(reinterpret_cast<uint4*>(&st_x[tau][0]) + c,
                           reinterpret_cast<const uint4*>(x + (size_t)(bos + tau) * cd + ch) + off);
            }
            if (cs_in) {
                const int per_q = QC * keep, tot = CH * (int)sizeof(T) * keep / 16;
                for (int c = tid; c < tot; c += kRecThreads) {
                    int ch, off;
                    range_of(c, per_q, ch, off);
                    cp_async16(reinterpret_cast<uint4*>(st_cs) + c,
                               reinterpret_cast<const uint4*>(cs_in + ((size_t)n * cd + ch) * keep) + off);
                }
            }
            {
                const int per_q = DK * K / 4, tot = CH * K / 4;
                for (int c = tid; c < tot; c += kRecThreads) {
                    int ch, off;
                    range_of(c, per_q, ch, off);
                    cp_async16(reinterpret_cast<uint4*>(st_w) + c,
                               reinterpret_cast<const uint4*>(p.conv_w + (size_t)ch * K) + off);
                }
            }
            constexpr int ZC = DV * (int)sizeof(T) / 16;
            for (int i = tid; i < m * ZC; i += kRecThreads) {
                const int tau = i / ZC, c = i - tau * ZC;
                cp_async16(reinterpret_cast<uint4*>(&st_z[tau][0]) + c,
                           reinterpret_cast<const uint4*>(z + ((size_t)(bos + tau) * hv_n + hv) * DV) + c);
            }
            cp_async_commit();
        }
        float a_pre = 0.f, b_pre = 0.f;
        if (tid < m) {
            const size_t gi = (size_t)(bos + tid) * hv_n + hv;
            a_pre = to_f32(av[gi]);
            b_pre = to_f32(bv[gi]);
        }

        // the state, from the copy in flight since the previous item; the next
        // item's copy goes out once every thread has taken its rows
        float4 s[RPT];
        if (!__syncthreads_and(tc::mbar_wait(&bar_s, s_phase))) {
            if (tid == 0) atomicCAS(&g_rec_error, 0, 30);
            cp_async_wait_all();
            break;
        }
        s_phase ^= 1;
        s_pending = false;
        {
            const float4* src = reinterpret_cast<const float4*>(s_next);
#pragma unroll
            for (int i = 0; i < RPT; ++i) s[i] = src[(RPT * rg + i) * L + c4];
        }
        __syncthreads();
        if (item + (int)gridDim.x < n_items) {
            if (tid == 0) issue_state(item + gridDim.x);
            s_pending = true;
        }

        // ---- conv + SiLU of the m tokens x (q | k | v) channels
        cp_async_wait_all();
        __syncthreads();
        if (K == 4) {
            // one channel a thread, sliding over the tokens: each input value
            // and the channel's weights are read once
            for (int lc = tid; lc < CH; lc += kRecThreads) {
                const float4 w4 = *reinterpret_cast<const float4*>(&st_w[lc * 4]);
                float h0 = 0.f, h1 = 0.f, h2 = 0.f;  // tokens -3, -2, -1
                if (cs_in) {
                    h0 = to_f32(st_cs[lc * 3]);
                    h1 = to_f32(st_cs[lc * 3 + 1]);
                    h2 = to_f32(st_cs[lc * 3 + 2]);
                }
                for (int tau = 0; tau < m; ++tau) {
                    const float xv = to_f32(st_x[tau][lc]);
                    float acc = fmaf(w4.x, h0, 0.f);
                    acc = fmaf(w4.y, h1, acc);
                    acc = fmaf(w4.z, h2, acc);
                    acc = fmaf(w4.w, xv, acc);
                    cbuf[tau][lc] = siluf_(acc);
                    h0 = h1;
                    h1 = h2;
                    h2 = xv;
                }
            }
        } else {
            for (int idx = tid; idx < m * CH; idx += kRecThreads) {
                const int tau = idx / CH, lc = idx % CH;
                float acc = 0.f;
                for (int j = 0; j < K; ++j) {
                    const int tt = tau - keep + j;
                    const float v = tt >= 0 ? to_f32(st_x[tt][lc])
                                    : cs_in ? to_f32(st_cs[lc * keep + keep + tt]) : 0.f;
                    acc = fmaf(st_w[lc * K + j], v, acc);
                }
                cbuf[tau][lc] = siluf_(acc);
            }
        }
        if (tid < m) {
            gam[tid] = expf(log_decay(a_pre, p.A_log[hv], p.dt_bias[hv], p.decay_form));
            bet[tid] = sigmoidf_(b_pre);
        }
        __syncthreads();

        // ---- per token (one warp each), from the raw conv outputs: the inverse
        // norms of q and k and, with each earlier token i, the products
        // k_i.k_i, k_i.k and k_i.q, turned into the coefficients of the solve
        if (warp < m) {
            constexpr int NV = 3 + 3 * (kRecSub - 1);
            const int tau = warp;
            float v[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j) v[j] = 0.f;
            for (int r = lane; r < DK; r += 32) {
                const float q = cbuf[tau][r], k = cbuf[tau][DK + r];
                v[0] = fmaf(q, q, v[0]);
                v[1] = fmaf(k, k, v[1]);
                v[2] = fmaf(k, q, v[2]);
#pragma unroll
                for (int j = 0; j < kRecSub - 1; ++j)
                    if (j < tau) {
                        const float ki = cbuf[j][DK + r];
                        v[3 + 3 * j] = fmaf(ki, ki, v[3 + 3 * j]);
                        v[4 + 3 * j] = fmaf(ki, k, v[4 + 3 * j]);
                        v[5 + 3 * j] = fmaf(ki, q, v[5 + 3 * j]);
                    }
            }
#pragma unroll
            for (int j = 0; j < NV; ++j)
                if (j < 3 + 3 * tau) v[j] = group_sum<32>(v[j]);
            if (lane == 0) {
                const float qi = rsqrtf(v[0] + p.l2_eps) * rsqrtf((float)DK);
                const float ki = rsqrtf(v[1] + p.l2_eps);
                nq[tau] = qi;
                nk[tau] = ki;
                cfq[tau][tau] = v[2] * ki * qi;
                float gc = gam[0];
                for (int u = 1; u <= tau; ++u) gc *= gam[u];
                gcum[tau] = gc;
                float dec = 1.f;  // decay over the tokens after j, through this one
#pragma unroll
                for (int j = kRecSub - 2; j >= 0; --j)
                    if (j < tau) {
                        dec *= gam[j + 1];
                        const float kj = rsqrtf(v[3 + 3 * j] + p.l2_eps);
                        cfk[tau][j] = dec * (v[4 + 3 * j] * kj * ki);
                        cfq[tau][j] = dec * (v[5 + 3 * j] * kj * qi);
                    }
            }
        }
        // ---- the one pass over the state (the conv has read the staging, which
        // the column sums now overwrite)
        switch (m) {
            case 1: ro_colsums<1, DK, DV, RPT, L, CH>(s, cbuf, rg, lane, warp, c4, red); break;
            case 2: ro_colsums<2, DK, DV, RPT, L, CH>(s, cbuf, rg, lane, warp, c4, red); break;
            case 3: ro_colsums<3, DK, DV, RPT, L, CH>(s, cbuf, rg, lane, warp, c4, red); break;
            default: ro_colsums<4, DK, DV, RPT, L, CH>(s, cbuf, rg, lane, warp, c4, red); break;
        }
        __syncthreads();

        // ---- the solve, two lanes a column: the even lane sums the key side
        // and forms delta_j, the odd lane the query side and o_j
        float o[kRecSub];
        if (tid < 2 * DV) {
            const int c = tid >> 1, h = tid & 1;
            float part[kRecSub], dl[kRecSub];
#pragma unroll
            for (int j = 0; j < kRecSub; ++j)
                if (j < m) {
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) acc += red[((w * kRecSub + j) * DV + c) * 2 + h];
                    part[j] = acc;
                }
#pragma unroll
            for (int j = 0; j < kRecSub; ++j)
                if (j < m) {
                    float kv = gcum[j] * (part[j] * nk[j]);
#pragma unroll
                    for (int i = 0; i < j; ++i) kv = fmaf(cfk[j][i], dl[i], kv);
                    const float d = bet[j] * (cbuf[j][2 * DK + c] - kv);
                    dl[j] = __shfl_sync(0xffffffffu, d, lane & ~1);
                    float oo = gcum[j] * (part[j] * nq[j]);
#pragma unroll
                    for (int i = 0; i <= j; ++i) oo = fmaf(cfq[j][i], dl[i], oo);
                    o[j] = oo;
                    const float o2 = group_sum<32>(h ? oo * oo : 0.f);
                    if (lane == 0) ysum[j][warp] = o2;
                }
        }
        __syncthreads();

        // ---- gated RMSNorm and the outputs: lane h of a column writes the
        // tokens j with j % 2 == h
        if (tid < 2 * DV) {
            const int c = tid >> 1, h = tid & 1;
            const float rn = p.norm_w[c];
#pragma unroll
            for (int j = 0; j < kRecSub; ++j)
                if (j < m) {
                    const float oj = __shfl_sync(0xffffffffu, o[j], lane | 1);
                    if ((j & 1) == h) {
                        float tot = 0.f;
#pragma unroll
                        for (int w = 0; w < 2 * DV / 32; ++w) tot += ysum[j][w];
                        const float rr = rsqrtf(tot / (float)DV + p.rms_eps);
                        const float zv = to_f32(st_z[j][c]);
                        out[(size_t)(bos + j) * hv_n * DV + (size_t)hv * DV + c] =
                            from_f32<T>(oj * rr * rn * gatef_(zv, p.act));
                    }
                }
        }
        __syncthreads();  // the staging and z rows are the next item's
    }

    // no copy may be in flight when the CTA leaves (only after a give-up)
    if (s_pending && tid == 0 && !tc::mbar_wait(&bar_s, s_phase)) atomicCAS(&g_rec_error, 0, 30);
}

// SMs of the current device, cached per device.
static int rec_sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (!cached[dev].load()) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cached[dev].store(n);
    }
    return cached[dev].load();
}

template <int DK, int DV, typename T, bool PC>
static cudaError_t launch_rec_inst(const RecurrentArgs& p, cudaStream_t st) {
    constexpr int kSmem = RecStage<DK, DV, T>::kBytes;  // the next item's state slab, the input staging
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
        cudaError_t e = cudaFuncSetAttribute(recurrent_kernel<DK, DV, T, PC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        // the whole unified L1 as shared memory: two CTAs per SM must fit
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(recurrent_kernel<DK, DV, T, PC>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true);
    }
    const int items = p.n_seq * p.n_v_heads;
    const int grid = std::min(items, kRecCtasPerSm * rec_sm_count());
    recurrent_kernel<DK, DV, T, PC><<<grid, kRecThreads, kSmem, st>>>(p);
    return cudaGetLastError();
}

template <int DK, int DV, typename T>
static cudaError_t launch_ro_inst(const RecurrentArgs& p, cudaStream_t st) {
    constexpr int kSmem = RoStage<DK, DV, T>::kBytes;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
        cudaError_t e = cudaFuncSetAttribute(verify_ro_kernel<DK, DV, T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(verify_ro_kernel<DK, DV, T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true);
    }
    const int items = p.n_seq * p.n_v_heads;
    const int grid = std::min(items, kRecCtasPerSm * rec_sm_count());
    verify_ro_kernel<DK, DV, T><<<grid, kRecThreads, kSmem, st>>>(p);
    return cudaGetLastError();
}

// A call the read-only kernel takes: no state written, a resident state read,
// at most kRecSub tokens in every sequence, scalar decay, 16-byte aligned
// inputs (its async copies), d_v <= 128.
static bool read_only_call(const RecurrentArgs& p, int dv) {
    const uintptr_t align = reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.z) |
                            reinterpret_cast<uintptr_t>(p.conv_w) |
                            reinterpret_cast<uintptr_t>(p.conv_state_in);
    return !p.state_out && !p.inter && p.state_in && !p.per_channel && !p.cu_seqlens && p.uniform_T >= 1 &&
           p.uniform_T <= kRecSub && dv <= 128 && (align & 15) == 0 && !std::getenv("GDN_VERIFY_TOKENWISE");
}

template <typename T>
static cudaError_t launch_recurrent_t(const RecurrentArgs& p, int dk, int dv, cudaStream_t st) {
    // the bulk state copies read 16-byte aligned slabs
    if (p.state_in && reinterpret_cast<uintptr_t>(p.state_in) % 16) return cudaErrorInvalidValue;
    if (read_only_call(p, dv)) {
#define GDN_RO_CASE(A, B) \
        if (dk == A && dv == B) return launch_ro_inst<A, B, T>(p, st);
        GDN_RO_CASE(32, 32) GDN_RO_CASE(32, 64) GDN_RO_CASE(32, 128)
        GDN_RO_CASE(64, 32) GDN_RO_CASE(64, 64) GDN_RO_CASE(64, 128)
        GDN_RO_CASE(128, 32) GDN_RO_CASE(128, 64) GDN_RO_CASE(128, 128)
#undef GDN_RO_CASE
    }
#define GDN_REC_CASE(A, B)                                                                         \
    if (dk == A && dv == B)                                                                        \
        return p.per_channel ? launch_rec_inst<A, B, T, true>(p, st) : launch_rec_inst<A, B, T, false>(p, st);
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

cudaError_t read_rec_error(int* code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_rec_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_rec_error, &zero, sizeof(int));
    }
    return e;
}

cudaError_t launch_commit_state(const CommitArgs& p, cudaStream_t st) {
    if (p.n_seq == 0) return cudaSuccess;
    commit_state_kernel<<<dim3(p.n_v_heads, p.n_seq), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
