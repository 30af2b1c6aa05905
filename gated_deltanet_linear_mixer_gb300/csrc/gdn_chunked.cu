// Chunked prefill of the gated delta rule on tcgen05 tensor cores (bf16
// operands, fp32 accumulation in tensor memory, fp32 state).
//
// The pages define the rule token by token (cherenkov qwen4_exp/cpu.rs fn
// deltanet; oxinfer 0.0.5 src/qwen.rs DeltaRule::run).  Unrolled over a chunk
// of C = 64 tokens that starts from state S0 it becomes dense algebra (the
// WY / UT form): with G_t the in-chunk cumulative log-decay,
//   A_ts = beta_t e^{G_t-G_s} k_t.k_s (s < t),  T = (I + A)^-1
//   W  = T diag(beta e^G) K,   U~ = T diag(beta) V,   U = U~ - W S0
//   O  = diag(e^G) Q S0 + (M o Q K^T) U,   M_ts = e^{G_t-G_s} (s <= t)
//   S1 = e^{G_last} S0 + (diag(e^{G_last-G}) K)^T U
// which equals the token recurrence in exact arithmetic.
//
// Kernels (after the prologue writes q_hat, k_hat, v, g, beta):
//   chunk_prep  one CTA per (chunk, key head), fully parallel: the Gram
//               products [Q;K] K^T on the tensor core, the masked decay
//               factors, the unit-lower-triangular inverse T in fp32 on CUDA
//               cores, then [W | U~] = T [beta e^G K | beta V] on the tensor
//               core, for each value head of the group.
//   chunk_scan  a 2-CTA cluster per (sequence, value head), each CTA owning
//               64 value lanes: carries S in fp32 registers across the chunks;
//               per chunk three MMA groups ([W; e^G Q] S, then (M o QK^T) U and
//               (e^{G_last-G} K)^T U), the state update and the fused gated
//               RMSNorm epilogue.
// Every operand tile is either loaded by TMA with the 128-byte swizzle or
// written by threads in the same layout.  B operands whose contraction runs
// along a tile's rows (S, U, [K|V] rows) use the MN-major descriptor; every A
// operand is K-major (the one A that would be MN-major, the scaled keys of the
// state increment, is transposed by threads).
#include <cstring>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
#include "gdn_tma_host.h"

namespace gdn {

using namespace tc;

constexpr int kC = 64;             // chunk length
constexpr int kD = 128;            // d_k = d_v on this path
constexpr int kChunkThreads = 256;

__device__ int g_device_error = 0;

__device__ __forceinline__ void report_error(int code) { atomicCAS(&g_device_error, 0, code); }

struct ChunkPos {
    int n, t0, L;
};

__device__ __forceinline__ ChunkPos chunk_pos(const int32_t* cu_seqlens, const int32_t* cu_chunks,
                                              int n_seq, int c) {
    const int n = seq_of_token(cu_chunks, n_seq, c);
    const int t0 = cu_seqlens[n] + (c - cu_chunks[n]) * kC;
    return {n, t0, min(kC, cu_seqlens[n + 1] - t0)};
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float f) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16) * f;
        const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * f;
        w[i] = pack_bf16x2(lo, hi);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Uniform decision after a bounded wait: every thread learns whether any
// thread's wait gave up.
__device__ __forceinline__ bool any_failed(bool ok) { return __syncthreads_or(ok ? 0 : 1) != 0; }

// ------------------------------------------------------------ chunk table
// cu_chunks[i] = sum over sequences j < i of ceil(len_j / C).  One CTA.
__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t* cu_seqlens, int n_seq,
                                                           int32_t* cu_chunks) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        cu_chunks[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < n_seq; base += 1024) {
        const int i = base + tid;
        const int v = i < n_seq ? (cu_seqlens[i + 1] - cu_seqlens[i] + kC - 1) / kC : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + carry;
        if (i < n_seq) cu_chunks[i + 1] = before + incl;
        __syncthreads();
        if (tid == 1023) carry = before + incl;
        __syncthreads();
    }
}

// Split arithmetic.  Every tensor-core operand is carried as a pair of bf16
// tiles, hi = bf16(x) and lo = bf16(x - hi), which together hold ~16
// significant bits; a product A.B is formed as hi.hi + hi.lo + lo.hi with
// fp32 accumulation (the dropped lo.lo term is ~2^-16 relative).  The gated
// outputs are heavy-tailed (up to ~50x their RMS), so plain bf16 operands
// (2^-9 relative) would put the largest outputs' error far above 2e-2 of the
// output RMS.
__device__ __forceinline__ void split_store(const float* f, uint8_t* hi, uint8_t* lo) {
    float h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        h[e] = __bfloat162float(__float2bfloat16_rn(f[e]));
        l[e] = f[e] - h[e];
    }
    *reinterpret_cast<uint4*>(hi) = pack_bf16x8(h);
    *reinterpret_cast<uint4*>(lo) = pack_bf16x8(l);
}
__device__ __forceinline__ void load_pair(const uint8_t* hi, const uint8_t* lo, float* f) {
    float l[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(hi), f);
    unpack_bf16x8(*reinterpret_cast<const uint4*>(lo), l);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] += l[e];
}
// D (+)= A.B with A, B given as (hi, lo) descriptor pairs.
__device__ __forceinline__ void mma3(uint32_t d, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl,
                                     uint32_t idesc, uint32_t accumulate) {
    mma_bf16(d, ah, bh, idesc, accumulate);
    mma_bf16(d, ah, bl, idesc, 1u);
    mma_bf16(d, al, bh, idesc, 1u);
}

// --------------------------------------------------------------- chunk_prep
constexpr uint32_t kPrepAgH = 0, kPrepAgL = 32768, kPrepTH = 65536, kPrepTL = 81920,
                   kPrepBH = 98304, kPrepBL = 131072, kPrepAt = 163840, kPrepVH = 180224,
                   kPrepVL = 196608, kPrepVec = 212992;

__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_prep_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                  ChunkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sAg[2] = {smem + kPrepAgH, smem + kPrepAgL};  // [Q; K] K-major (hi, lo)
    uint8_t* sT[2] = {smem + kPrepTH, smem + kPrepTL};     // T K-major, rows 64.. zero
    uint8_t* sB[2] = {smem + kPrepBH, smem + kPrepBL};     // [beta e^G K | beta V] MN-major
    float* sAt = reinterpret_cast<float*>(smem + kPrepAt); // A^T [s][t] of one head
    uint8_t* sV[2] = {smem + kPrepVH, smem + kPrepVL};     // v rows of one head (hi, lo)
    const int R = p.n_v_heads / p.n_k_heads;
    float* sG = reinterpret_cast<float*>(smem + kPrepVec);
    float* sBeta = sG + R * kC;
    __shared__ __align__(8) uint64_t bar_tma, bar_mma, bar_v;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, hk = blockIdx.y;
    const int hv_n = p.n_v_heads;
    const int cd = 2 * p.n_k_heads * kD + hv_n * kD;
    const ChunkPos cp = chunk_pos(p.cu_seqlens, p.cu_chunks, p.n_seq, c);
    const int t0 = cp.t0, L = cp.L;

    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_v, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 512);
    for (int i = tid; i < 1024; i += kChunkThreads)
        reinterpret_cast<uint4*>(sT[i >> 9] + 8192)[i & 511] = make_uint4(0u, 0u, 0u, 0u);
    if (warp < R) {  // cumulative log-decay and write strength of value head hk*R + warp
        const int h = hk * R + warp;
        const int s0 = 2 * lane, s1 = 2 * lane + 1;
        float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
        if (s0 < L) {
            g0 = p.g[(size_t)(t0 + s0) * hv_n + h];
            b0 = p.beta[(size_t)(t0 + s0) * hv_n + h];
        }
        if (s1 < L) {
            g1 = p.g[(size_t)(t0 + s1) * hv_n + h];
            b1 = p.beta[(size_t)(t0 + s1) * hv_n + h];
        }
        const float local = g0 + g1;
        float incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const float excl = incl - local;
        sG[warp * kC + s0] = excl + g0;
        sG[warp * kC + s1] = excl + g0 + g1;
        sBeta[warp * kC + s0] = b0;
        sBeta[warp * kC + s1] = b1;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;        // cols 0..255: [W | U~]
    const uint32_t tmem_g = tmem + 256;     // cols 256..319: Gram
    uint32_t mma_phase = 0;
    bool tma_pending = false, mma_pending = false;
    int v_issued = 0, v_done = 0;  // value heads whose v tiles were requested / consumed
    // v rows of value head hk*R + r (both column blocks, hi and lo) -> sV
    auto issue_v = [&](int r) {
        const int vc = 2 * p.n_k_heads * kD + (hk * R + r) * kD;
        mbar_arrive_expect_tx(&bar_v, 4 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_2d(sV[0] + b * 8192, &map_qh, &bar_v, vc + 64 * b, t0);
            tma_load_2d(sV[1] + b * 8192, &map_ql, &bar_v, vc + 64 * b, t0);
        }
    };

    do {
        if (tid == 0) {
            issue_v(0);
            mbar_arrive_expect_tx(&bar_tma, 8 * 8192);
            const int qc = hk * kD, kc = p.n_k_heads * kD + hk * kD;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tma_load_2d(sAg[0] + b * 16384, &map_qh, &bar_tma, qc + 64 * b, t0);
                tma_load_2d(sAg[0] + b * 16384 + 8192, &map_qh, &bar_tma, kc + 64 * b, t0);
                tma_load_2d(sAg[1] + b * 16384, &map_ql, &bar_tma, qc + 64 * b, t0);
                tma_load_2d(sAg[1] + b * 16384 + 8192, &map_ql, &bar_tma, kc + 64 * b, t0);
            }
        }
        tma_pending = true;
        v_issued = 1;
        if (any_failed(mbar_wait(&bar_tma, 0))) {
            if (tid == 0) report_error(1);
            break;
        }
        tma_pending = false;
        if (L < kC) {  // rows past the chunk belong to another sequence: zero them
            const int nr = kC - L;
            for (int i = tid; i < nr * 64; i += kChunkThreads) {
                const int ch = i & 7, rest = i >> 3;
                const int r = L + rest % nr, pb = rest / nr;  // pb: hi/lo x part x block
                *reinterpret_cast<uint4*>(sAg[pb >> 2] + ((pb >> 1) & 1) * 16384 +
                                          ((pb & 1) * 64 + r) * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (tid == 0) {  // Gram: rows 0..63 = Q K^T, rows 64..127 = K K^T
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                const uint32_t ah = smem_u32(sAg[0]) + off, al = smem_u32(sAg[1]) + off;
                mma3(tmem_g, desc_kmajor_sw128(ah), desc_kmajor_sw128(al),
                     desc_kmajor_sw128(ah + 8192), desc_kmajor_sw128(al + 8192),
                     idesc_bf16_f32(128, 64), k > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        if (any_failed(mbar_wait(&bar_mma, mma_phase))) {
            if (tid == 0) report_error(2);
            break;
        }
        mma_pending = false;
        mma_phase ^= 1;
        tc_fence_after_sync();

        bool failed = false;
        for (int r = 0; r < R; ++r) {
            const int h = hk * R + r;
            const float* Gr = sG + r * kC;
            const float* Br = sBeta + r * kC;
            if (any_failed(mbar_wait(&bar_v, r & 1))) {  // this head's v tiles
                if (tid == 0) report_error(7);
                failed = true;
                break;
            }
            v_done = r + 1;
            if (warp < 4) {
                float v[64];
                tmem_ld32(tmem_g + ((32u * warp) << 16), v);
                tmem_ld32(tmem_g + ((32u * warp) << 16) + 32, v + 32);
                if (warp < 2) {  // masked decayed Q K^T row t -> workspace (hi, lo)
                    const int t = 32 * warp + lane;
                    const float Gt = Gr[t];
                    const size_t o = ((size_t)(c * hv_n + h) * kC + t) * kC;
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int s = q8 * 8 + e;
                            f[e] = s <= t ? expf(Gt - Gr[s]) * v[s] : 0.f;
                        }
                        split_store(f, reinterpret_cast<uint8_t*>(p.qk_hi + o + 8 * q8),
                                    reinterpret_cast<uint8_t*>(p.qk_lo + o + 8 * q8));
                    }
                } else {  // A = strictly-lower beta_t e^{G_t-G_s} k_t.k_s, stored transposed
                    const int t = 32 * (warp - 2) + lane;
                    const float Gt = Gr[t], bt = Br[t];
#pragma unroll
                    for (int s = 0; s < kC; ++s)
                        sAt[s * kC + t] = s < t ? bt * expf(Gt - Gr[s]) * v[s] : 0.f;
                }
            } else {
                // B rows s: [beta_s e^{G_s} k_s | beta_s v_s], MN-major, hi/lo
                for (int it = tid - 128; it < kC * 32; it += 128) {
                    const int ch = it & 7, blk = (it >> 3) & 3, s = it >> 5;
                    const uint32_t pos = static_cast<uint32_t>((ch ^ (s & 7)) << 4);
                    const float bt = Br[s];
                    float f[8];
                    if (blk < 2) {
                        const uint32_t so = blk * 16384 + (64 + s) * 128 + pos;
                        load_pair(sAg[0] + so, sAg[1] + so, f);
                        const float sc = bt * expf(Gr[s]);
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] *= sc;
                    } else if (s < L) {
                        const uint32_t so = (blk - 2) * 8192 + s * 128 + pos;
                        load_pair(sV[0] + so, sV[1] + so, f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] *= bt;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = 0.f;
                    }
                    split_store(f, sB[0] + blk * 8192 + s * 128 + pos, sB[1] + blk * 8192 + s * 128 + pos);
                }
            }
            __syncthreads();
            if (tid == 0 && r + 1 < R) {  // next head's v tiles land during this head's solve
                issue_v(r + 1);
                v_issued = r + 2;
            }
            if (warp >= 2 && warp < 4) {
                // operand rows the state scan needs, prepared here off its chain:
                // q~_t = e^{G_t} q_t (zero past the chunk), hi/lo
                const int t = 32 * (warp - 2) + lane;
                const float f = t < L ? expf(Gr[t]) : 0.f;
                const size_t o = ((size_t)(c * hv_n + h) * kC + t) * kD;
#pragma unroll
                for (int ch = 0; ch < 16; ++ch) {
                    const uint32_t so = (ch >> 3) * 16384 + t * 128 + (((ch & 7) ^ (t & 7)) << 4);
                    float v[8];
                    load_pair(sAg[0] + so, sAg[1] + so, v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = t < L ? v[e] * f : 0.f;
                    split_store(v, reinterpret_cast<uint8_t*>(p.qt_hi + o + 8 * ch),
                                reinterpret_cast<uint8_t*>(p.qt_lo + o + 8 * ch));
                }
            } else if (warp >= 4) {
                // (e^{G_last-G_s} k_s)^T: thread i writes key lane i over the tokens
                const int ki = tid - 128;
                const float GL = Gr[L - 1];
                const uint32_t col = (ki >> 6) * 16384 + (ki & 7) * 2;
                const uint32_t chunk = (ki & 63) >> 3;
                const size_t o = ((size_t)(c * hv_n + h) * kD + ki) * kC;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int sidx = 8 * c8 + e;
                        const uint32_t so = col + (64 + sidx) * 128 + ((chunk ^ (sidx & 7)) << 4);
                        const float kv =
                            __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sAg[0] + so)) +
                            __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sAg[1] + so));
                        v[e] = sidx < L ? kv * expf(GL - Gr[sidx]) : 0.f;
                    }
                    split_store(v, reinterpret_cast<uint8_t*>(p.kt_hi + o + 8 * c8),
                                reinterpret_cast<uint8_t*>(p.kt_lo + o + 8 * c8));
                }
            }
            if (warp < 2) {
                // T = (I + A)^-1: thread j solves (I + A) x = e_j by forward
                // substitution, eliminating one known entry at a time.
                const int j = tid;
                float x[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) x[t] = t == j ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < kC - 1; ++s) {
                    const float xs = x[s];
#pragma unroll
                    for (int t = s + 1; t < kC; ++t) x[t] = fmaf(-sAt[s * kC + t], xs, x[t]);
                }
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    const uint32_t o = t * 128 + ((((j >> 3) ^ (t & 7))) << 4) + (j & 7) * 2;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(x[t]);
                    *reinterpret_cast<__nv_bfloat16*>(sT[0] + o) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(sT[1] + o) =
                        __float2bfloat16_rn(x[t] - __bfloat162float(hi));
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
            if (tid == 0) {  // W = T beta e^G K (cols 0..127), U~ = T beta V (cols 128..255)
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma3(tmem + 128 * half, desc_kmajor_sw128(smem_u32(sT[0]) + k * 32),
                             desc_kmajor_sw128(smem_u32(sT[1]) + k * 32),
                             desc_mnmajor_sw128(smem_u32(sB[0]) + half * 16384 + k * 2048, 8192),
                             desc_mnmajor_sw128(smem_u32(sB[1]) + half * 16384 + k * 2048, 8192),
                             idesc_bf16_f32(128, 128, false, true), k > 0 ? 1u : 0u);
                mma_commit(&bar_mma);
            }
            mma_pending = true;
            if (any_failed(mbar_wait(&bar_mma, mma_phase))) {
                if (tid == 0) report_error(3);
                failed = true;
                break;
            }
            mma_pending = false;
            mma_phase ^= 1;
            tc_fence_after_sync();
            if ((warp & 3) < 2) {  // rows t of W (warps 0,1, hi/lo) and of U~ (warps 4,5, fp32)
                const int t = 32 * (warp & 3) + lane;
                const size_t o = ((size_t)(c * hv_n + h) * kC + t) * kD;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    float v[32];
                    tmem_ld32(tmem + ((32u * (warp & 3)) << 16) + (warp >> 2) * 128 + 32 * cb, v);
                    if (warp < 4) {
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8)
                            split_store(v + 8 * q8,
                                        reinterpret_cast<uint8_t*>(p.w_hi + o + 32 * cb + 8 * q8),
                                        reinterpret_cast<uint8_t*>(p.w_lo + o + 32 * cb + 8 * q8));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(p.u_ws + o + 32 * cb);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                    }
                }
            }
            if (tid < kC) p.gcum_ws[(size_t)(c * hv_n + h) * kC + tid] = Gr[tid];
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
        }
        (void)failed;
    } while (false);

    // Unwind after a give-up: let in-flight copies and MMAs land first.
    v_issued = __syncthreads_or(v_issued > v_done) ? v_done + 1 : v_done;
    if (tma_pending) mbar_wait(&bar_tma, 0);
    if (v_issued > v_done) mbar_wait(&bar_v, v_done & 1);
    if (mma_pending) mbar_wait(&bar_mma, mma_phase);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// --------------------------------------------------------------- chunk_scan
// A cluster of kSplit CTAs shares one (sequence, value head): CTA p owns value
// lanes [64p, 64p+64) of the state, the outputs and U.  The per-token sums of
// squares of the gated RMSNorm are exchanged through distributed shared memory.
constexpr int kSplit = 2;
constexpr int kDS = kD / kSplit;   // value lanes per CTA
constexpr uint32_t kScanBsH = 0, kScanBsL = 16384, kScanAwH = 32768, kScanAwL = 65536,
                   kScanAqH = 98304, kScanAqL = 114688, kScanBuH = 131072, kScanBuL = 139264,
                   kScanAkH = 147456, kScanAkL = 163840, kScanEnd = 180224;

__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kChunkThreads, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap map_qth, const __grid_constant__ CUtensorMap map_qtl,
                  const __grid_constant__ CUtensorMap map_wh, const __grid_constant__ CUtensorMap map_wl,
                  const __grid_constant__ CUtensorMap map_kqh, const __grid_constant__ CUtensorMap map_kql,
                  const __grid_constant__ CUtensorMap map_kth, const __grid_constant__ CUtensorMap map_ktl,
                  ChunkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sBs[2] = {smem + kScanBsH, smem + kScanBsL};  // S slice, MN-major 128 x 64
    uint8_t* sAw[2] = {smem + kScanAwH, smem + kScanAwL};  // [W; e^G Q] K-major 128 x 128
    uint8_t* sAq[2] = {smem + kScanAqH, smem + kScanAqL};  // [0; M o QK^T] K-major 128 x 64
    uint8_t* sBu[2] = {smem + kScanBuH, smem + kScanBuL};  // U slice, MN-major 64 x 64
    uint8_t* sAk[2] = {smem + kScanAkH, smem + kScanAkL};  // (e^{G_last-G} K)^T, K-major 128 x 64
    __shared__ float sSsq[2][kC];
    __shared__ float sSsqC[2][kC];
    __shared__ __align__(8) uint64_t bar_wq, bar_k, bar_kq, bar_mma;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hf = warp >> 2;
    const int row = 32 * q + lane;  // tensor-memory lane this thread reads
    const uint32_t rank = cluster_ctarank();
    const int h = blockIdx.x / kSplit, n = blockIdx.y;
    const int j0 = static_cast<int>(rank) * kDS + 32 * hf;  // first value lane of this thread
    const int hv_n = p.n_v_heads;
    const int R = hv_n / p.n_k_heads, hk = h / R;
    const int bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    const int c_begin = p.cu_chunks[n], n_ch = p.cu_chunks[n + 1] - c_begin;
    const size_t slab = ((size_t)n * hv_n + h) * kD * kD;

    // fp32 state: this thread owns S[row][j0 .. j0+31]
    float S[32];
    if (p.state_in) {
        const float4* src = reinterpret_cast<const float4*>(p.state_in + slab + (size_t)row * kD + j0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = src[i];
            S[4 * i] = v.x; S[4 * i + 1] = v.y; S[4 * i + 2] = v.z; S[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) S[i] = 0.f;
    }
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const uint32_t o = row * 128 + (((4 * hf + ch) ^ (row & 7)) << 4);
        split_store(S + 8 * ch, sBs[0] + o, sBs[1] + o);
    }
    for (int i = tid; i < 1024; i += kChunkThreads)
        reinterpret_cast<uint4*>(sAq[i >> 9])[i & 511] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        mbar_init(&bar_wq, 1);
        mbar_init(&bar_k, 1);
        mbar_init(&bar_kq, 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 128);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;     // cols 0..63: [W S ; e^G Q S + (M o QK^T) U]
    const uint32_t tmem_s = tmem + 64;   // cols 64..127: K'^T U
    const uint32_t lane_off = (32u * q) << 16;
    const uint32_t peer_ssq = map_to_rank(smem_u32(&sSsqC[0][0]), rank ^ 1u);
    const bool sigmoid_gate = p.act == 1;
    const uint32_t id_p4 = idesc_bf16_f32(128, kDS, false, true);
    // in-chunk log-decay at the chunk's last token, e^{.} of which decays the state
    auto last_g = [&](int i) {
        const int L = min(kC, eos - (bos + i * kC));
        return p.gcum_ws[(size_t)((c_begin + i) * hv_n + h) * kC + L - 1];
    };

    // Loads of chunk i (within this sequence), three groups with their own
    // barriers so that each can be issued as soon as its buffer is free.
    auto issue_wq = [&](int i) {  // W rows and e^{G} q rows -> [W; Q~]
        const int wrow = ((c_begin + i) * hv_n + h) * kC;
        mbar_arrive_expect_tx(&bar_wq, 8 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_2d(sAw[0] + b * 16384, &map_wh, &bar_wq, 64 * b, wrow);
            tma_load_2d(sAw[1] + b * 16384, &map_wl, &bar_wq, 64 * b, wrow);
            tma_load_2d(sAw[0] + b * 16384 + 8192, &map_qth, &bar_wq, 64 * b, wrow);
            tma_load_2d(sAw[1] + b * 16384 + 8192, &map_qtl, &bar_wq, 64 * b, wrow);
        }
    };
    auto issue_k = [&](int i) {  // (e^{G_last-G} K)^T rows -> A of the state increment
        const int krow = ((c_begin + i) * hv_n + h) * kD;
        mbar_arrive_expect_tx(&bar_k, 4 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_2d(sAk[0] + b * 8192, &map_kth, &bar_k, 0, krow + 64 * b);
            tma_load_2d(sAk[1] + b * 8192, &map_ktl, &bar_k, 0, krow + 64 * b);
        }
    };
    auto issue_kq = [&](int i) {  // masked decayed Q K^T -> rows 64..127 of [0; M o QK^T]
        const int wrow = ((c_begin + i) * hv_n + h) * kC;
        mbar_arrive_expect_tx(&bar_kq, 2 * 8192);
        tma_load_2d(sAq[0] + 8192, &map_kqh, &bar_kq, 0, wrow);
        tma_load_2d(sAq[1] + 8192, &map_kql, &bar_kq, 0, wrow);
    };
    // issued[g] / done[g]: loads of each group requested / waited for
    int issued_wq = 0, issued_k = 0, issued_kq = 0, done_wq = 0, done_k = 0, done_kq = 0;
    uint32_t mma_phase = 0;
    bool mma_pending = false, dead = false;
    if (n_ch > 0) {
        if (tid == 0) {
            issue_wq(0);
            issue_k(0);
            issue_kq(0);
        }
        issued_wq = issued_k = issued_kq = 1;
    }
    float gl_cur = n_ch > 0 ? last_g(0) : 0.f, gl_next = 0.f;
    float ut[32];  // U~ row `row`, value lanes j0..j0+31, of the current chunk (q < 2)
    if (q < 2 && n_ch > 0) {
        const float4* src = reinterpret_cast<const float4*>(p.u_ws + ((size_t)(c_begin * hv_n + h) * kC + row) * kD + j0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = src[i];
            ut[4 * i] = v.x; ut[4 * i + 1] = v.y; ut[4 * i + 2] = v.z; ut[4 * i + 3] = v.w;
        }
    }

    for (int i = 0; i < n_ch; ++i) {
        const int t0 = bos + i * kC;
        const int L = min(kC, eos - t0);
        const int buf = i & 1;
        const float GL = gl_cur;
        uint4 zr[4];
        do {
            if (dead) break;
            if (i + 1 < n_ch) gl_next = last_g(i + 1);  // prefetched for the next chunk
            if (q >= 2 && row - 64 < L) {  // this chunk's z rows for the epilogue
                const uint4* zp = reinterpret_cast<const uint4*>(
                    p.z + (size_t)(t0 + row - 64) * hv_n * kD + (size_t)h * kD + j0);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) zr[ch] = zp[ch];
            }
            const bool okk = mbar_wait(&bar_k, i & 1);
            const bool okw = mbar_wait(&bar_wq, i & 1);
            if (any_failed(okk && okw)) {
                if (tid == 0) report_error(4);
                dead = true;
                break;
            }
            done_k = done_wq = i + 1;
            tc_fence_after_sync();
            if (tid == 0) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // [W S ; e^G Q S]
                    const uint32_t ao = (k >> 2) * 16384 + (k & 3) * 32;
                    mma3(tmem, desc_kmajor_sw128(smem_u32(sAw[0]) + ao),
                         desc_kmajor_sw128(smem_u32(sAw[1]) + ao),
                         desc_mnmajor_sw128(smem_u32(sBs[0]) + k * 2048, 16384),
                         desc_mnmajor_sw128(smem_u32(sBs[1]) + k * 2048, 16384), id_p4,
                         k > 0 ? 1u : 0u);
                }
                mma_commit(&bar_mma);
            }
            mma_pending = true;
            if (any_failed(mbar_wait(&bar_mma, mma_phase))) {
                if (tid == 0) report_error(5);
                dead = true;
                break;
            }
            mma_pending = false;
            mma_phase ^= 1;
            tc_fence_after_sync();
            if (tid == 0 && i + 1 < n_ch) issue_wq(i + 1);  // [W; Q] consumed
            if (i + 1 < n_ch) issued_wq = i + 2;
            if (q < 2) {  // U = U~ - W S for token row `row`, value lanes j0..j0+31
                float ws[32];
                tmem_ld32(tmem + lane_off + 32 * hf, ws);
#pragma unroll
                for (int e = 0; e < 32; ++e) ut[e] -= ws[e];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t o = row * 128 + (((4 * hf + ch) ^ (row & 7)) << 4);
                    split_store(ut + 8 * ch, sBu[0] + o, sBu[1] + o);
                }
                if (i + 1 < n_ch) {  // next chunk's U~ row
                    const float4* src = reinterpret_cast<const float4*>(
                        p.u_ws + ((size_t)((c_begin + i + 1) * hv_n + h) * kC + row) * kD + j0);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float4 v = src[e];
                        ut[4 * e] = v.x; ut[4 * e + 1] = v.y; ut[4 * e + 2] = v.z; ut[4 * e + 3] = v.w;
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            const bool okq = mbar_wait(&bar_kq, i & 1);
            if (any_failed(okq)) {
                if (tid == 0) report_error(8);
                dead = true;
                break;
            }
            done_kq = i + 1;
            tc_fence_after_sync();
            if (tid == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // O += (M o QK^T) U   (rows 0..63 of A are zero)
                    const uint64_t bh = desc_mnmajor_sw128(smem_u32(sBu[0]) + k * 2048, 8192);
                    const uint64_t bl = desc_mnmajor_sw128(smem_u32(sBu[1]) + k * 2048, 8192);
                    mma3(tmem, desc_kmajor_sw128(smem_u32(sAq[0]) + k * 32),
                         desc_kmajor_sw128(smem_u32(sAq[1]) + k * 32), bh, bl, id_p4, 1u);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // state increment (e^{G_last-G} K)^T U
                    const uint64_t bh = desc_mnmajor_sw128(smem_u32(sBu[0]) + k * 2048, 8192);
                    const uint64_t bl = desc_mnmajor_sw128(smem_u32(sBu[1]) + k * 2048, 8192);
                    mma3(tmem_s, desc_kmajor_sw128(smem_u32(sAk[0]) + k * 32),
                         desc_kmajor_sw128(smem_u32(sAk[1]) + k * 32), bh, bl, id_p4,
                         k > 0 ? 1u : 0u);
                }
                mma_commit(&bar_mma);
            }
            mma_pending = true;
            if (any_failed(mbar_wait(&bar_mma, mma_phase))) {
                if (tid == 0) report_error(6);
                dead = true;
                break;
            }
            mma_pending = false;
            mma_phase ^= 1;
            tc_fence_after_sync();
            if (tid == 0 && i + 1 < n_ch) {  // [0; M o QK^T] and the keys are consumed
                issue_kq(i + 1);
                issue_k(i + 1);
            }
            if (i + 1 < n_ch) issued_kq = issued_k = i + 2;
            {  // S <- e^{G_last} S + K'^T U ; refresh the split copy
                const float gam = expf(GL);
                float ds[32];
                tmem_ld32(tmem_s + lane_off + 32 * hf, ds);
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] = fmaf(gam, S[j], ds[j]);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t o = row * 128 + (((4 * hf + ch) ^ (row & 7)) << 4);
                    split_store(S + 8 * ch, sBs[0] + o, sBs[1] + o);
                }
            }
            if (q >= 2) {  // output rows: partial sum of squares over 32 value lanes
                float o[32];
                tmem_ld32(tmem + lane_off + 32 * hf, o);
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) ss = fmaf(o[j], o[j], ss);
                sSsq[hf][row - 64] = ss;
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
            if (tid < kC) sSsqC[buf][tid] = sSsq[0][tid] + sSsq[1][tid];
        } while (false);
        gl_cur = gl_next;
        // Exchange the CTA's partial sums with its peer; every CTA of the
        // cluster passes this barrier once per chunk, also after an error.
        cluster_arrive();
        cluster_wait();
        if (!dead && q >= 2) {  // gated RMSNorm epilogue for token t, value lanes j0..j0+31
            const int t = row - 64;
            float o[32];
            tmem_ld32(tmem + lane_off + 32 * hf, o);  // warp-collective: every lane loads
            if (t < L) {
                const float tot = sSsqC[buf][t] + ld_cluster_f32(peer_ssq + (uint32_t)(buf * kC + t) * 4u);
                const float rr = rsqrtf(tot * (1.f / kD) + p.rms_eps);
                uint4* op = reinterpret_cast<uint4*>(p.out + (size_t)(t0 + t) * hv_n * kD + (size_t)h * kD + j0);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    float zz[8], y[8];
                    unpack_bf16x8(zr[ch], zz);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float gate = sigmoid_gate ? sigmoidf_(zz[e]) : siluf_(zz[e]);
                        y[e] = o[8 * ch + e] * rr * p.norm_w[j0 + 8 * ch + e] * gate;
                    }
                    op[ch] = pack_bf16x8(y);
                }
            }
            tc_fence_before_sync();
        }
    }

    // Unwind: let every copy and MMA still in flight land before leaving.
    if (__syncthreads_or(issued_k > done_k)) mbar_wait(&bar_k, done_k & 1);
    if (__syncthreads_or(issued_wq > done_wq)) mbar_wait(&bar_wq, done_wq & 1);
    if (__syncthreads_or(issued_kq > done_kq)) mbar_wait(&bar_kq, done_kq & 1);
    if (mma_pending) mbar_wait(&bar_mma, mma_phase);
    if (p.state_out) {
        float4* dst = reinterpret_cast<float4*>(p.state_out + slab + (size_t)row * kD + j0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    }
    // No CTA may leave while its peer can still read its shared memory.
    cluster_arrive();
    cluster_wait();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------- host
size_t chunked_workspace_bytes(int n_seq, const int32_t* cu_host, int n_k_heads, int n_v_heads,
                               ChunkLayout* lay) {
    ChunkLayout l{};
    const int T = n_seq > 0 ? cu_host[n_seq] : 0;
    long long chunks = 0;
    for (int i = 0; i < n_seq; ++i) chunks += (cu_host[i + 1] - cu_host[i] + kC - 1) / kC;
    const size_t cd = 2 * (size_t)n_k_heads * kD + (size_t)n_v_heads * kD;
    const size_t crow = (size_t)chunks * n_v_heads * kC;  // rows of the per-chunk arrays
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    size_t off = 0;
    // q|k|v rows are padded by one chunk so that every 64-row TMA box that
    // starts inside the batch stays inside the tensor (no out-of-bounds boxes).
    l.qkv_hi = off; off = up(off + ((size_t)T + kC) * cd * 2);
    l.qkv_lo = off; off = up(off + ((size_t)T + kC) * cd * 2);
    l.g = off; off = up(off + (size_t)T * n_v_heads * 4);
    l.beta = off; off = up(off + (size_t)T * n_v_heads * 4);
    l.cu_chunks = off; off = up(off + (size_t)(n_seq + 1) * 4);
    l.w_hi = off; off = up(off + crow * kD * 2);
    l.w_lo = off; off = up(off + crow * kD * 2);
    l.u = off; off = up(off + crow * kD * 4);
    l.qk_hi = off; off = up(off + crow * kC * 2);
    l.qk_lo = off; off = up(off + crow * kC * 2);
    l.qt_hi = off; off = up(off + crow * kD * 2);
    l.qt_lo = off; off = up(off + crow * kD * 2);
    l.kt_hi = off; off = up(off + (size_t)chunks * n_v_heads * kD * kC * 2);
    l.kt_lo = off; off = up(off + (size_t)chunks * n_v_heads * kD * kC * 2);
    l.gcum = off; off = up(off + crow * 4);
    l.total = off;
    l.n_chunks = static_cast<int>(chunks);
    if (lay) *lay = l;
    return off;
}

cudaError_t launch_chunked_prefill(const ChunkLaunch& a, cudaStream_t st) {
    const ChunkLayout& l = a.layout;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const int hk_n = a.n_k_heads, hv_n = a.n_v_heads;
    const int cd = 2 * hk_n * kD + hv_n * kD;
    const int T = a.n_tokens;
    const int R = hv_n / hk_n;

    // 1. prologue: conv + SiLU + L2 norm + gates -> q|k|v (hi, lo), g, beta
    ConvArgs cv{};
    cv.n_seq = a.n_seq; cv.n_tokens = T; cv.n_k_heads = hk_n; cv.n_v_heads = hv_n;
    cv.d_k = kD; cv.d_v = kD; cv.conv_k = a.conv_k; cv.l2_eps = a.l2_eps;
    cv.cu_seqlens = a.cu_seqlens; cv.x = a.x; cv.a = a.a; cv.b = a.b;
    cv.conv_w = a.conv_w; cv.A_log = a.A_log; cv.dt_bias = a.dt_bias;
    cv.conv_state_in = a.conv_state_in;
    cv.qkv_out = ws + l.qkv_hi;
    cv.qkv_lo_out = ws + l.qkv_lo;
    cv.g_out = reinterpret_cast<float*>(ws + l.g);
    cv.beta_out = reinterpret_cast<float*>(ws + l.beta);
    cudaError_t e = timed_launch("conv_prologue", st, [&] { return launch_conv_prologue(cv, true, st); });
    if (e != cudaSuccess) return e;
    if (a.n_seq == 0) return cudaSuccess;

    int32_t* cu_chunks = reinterpret_cast<int32_t*>(ws + l.cu_chunks);
    e = timed_launch("chunk_table", st, [&] {
        chunk_table_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.n_seq, cu_chunks);
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;

    ChunkArgs p{};
    p.n_seq = a.n_seq; p.n_tokens = T; p.n_chunks = l.n_chunks;
    p.n_k_heads = hk_n; p.n_v_heads = hv_n; p.act = a.act; p.rms_eps = a.rms_eps;
    p.cu_seqlens = a.cu_seqlens; p.cu_chunks = cu_chunks;
    p.qkv_hi = reinterpret_cast<const __nv_bfloat16*>(ws + l.qkv_hi);
    p.qkv_lo = reinterpret_cast<const __nv_bfloat16*>(ws + l.qkv_lo);
    p.g = reinterpret_cast<const float*>(ws + l.g);
    p.beta = reinterpret_cast<const float*>(ws + l.beta);
    p.z = static_cast<const __nv_bfloat16*>(a.z);
    p.norm_w = a.norm_w;
    p.state_in = a.state_in; p.state_out = a.state_out;
    p.w_hi = reinterpret_cast<__nv_bfloat16*>(ws + l.w_hi);
    p.w_lo = reinterpret_cast<__nv_bfloat16*>(ws + l.w_lo);
    p.u_ws = reinterpret_cast<float*>(ws + l.u);
    p.qk_hi = reinterpret_cast<__nv_bfloat16*>(ws + l.qk_hi);
    p.qk_lo = reinterpret_cast<__nv_bfloat16*>(ws + l.qk_lo);
    p.qt_hi = reinterpret_cast<__nv_bfloat16*>(ws + l.qt_hi);
    p.qt_lo = reinterpret_cast<__nv_bfloat16*>(ws + l.qt_lo);
    p.kt_hi = reinterpret_cast<__nv_bfloat16*>(ws + l.kt_hi);
    p.kt_lo = reinterpret_cast<__nv_bfloat16*>(ws + l.kt_lo);
    p.gcum_ws = reinterpret_cast<float*>(ws + l.gcum);
    p.out = static_cast<__nv_bfloat16*>(a.out);

    // Tensor maps; with no chunk at all (only empty sequences) no kernel
    // dereferences them and they stay zero.
    CUtensorMap m_qh, m_ql, m_wh, m_wl, m_kqh, m_kql, m_qth, m_qtl, m_kth, m_ktl;
    std::memset(&m_qh, 0, sizeof(m_qh));
    m_ql = m_wh = m_wl = m_kqh = m_kql = m_qth = m_qtl = m_kth = m_ktl = m_qh;
    const uint64_t crow = (uint64_t)l.n_chunks * hv_n * kC;
    if (l.n_chunks > 0) {
        if (!make_tma_map_bf16_2d(&m_qh, ws + l.qkv_hi, (uint64_t)T + kC, cd, cd, 64, 64) ||
            !make_tma_map_bf16_2d(&m_ql, ws + l.qkv_lo, (uint64_t)T + kC, cd, cd, 64, 64) ||
            !make_tma_map_bf16_2d(&m_wh, ws + l.w_hi, crow, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_wl, ws + l.w_lo, crow, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kqh, ws + l.qk_hi, crow, kC, kC, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kql, ws + l.qk_lo, crow, kC, kC, 64, 64) ||
            !make_tma_map_bf16_2d(&m_qth, ws + l.qt_hi, crow, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_qtl, ws + l.qt_lo, crow, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kth, ws + l.kt_hi, (uint64_t)l.n_chunks * hv_n * kD, kC, kC, 64, 64) ||
            !make_tma_map_bf16_2d(&m_ktl, ws + l.kt_lo, (uint64_t)l.n_chunks * hv_n * kD, kC, kC, 64, 64))
            return cudaErrorInvalidValue;
    }

    const size_t prep_smem = 1024 + kPrepVec + (size_t)R * 2 * kC * 4;
    const size_t scan_smem = 1024 + kScanEnd;
    static bool attrs_set = false;
    if (!attrs_set) {
        cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(1024 + kPrepVec + 8 * 2 * kC * 4));
        cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(scan_smem));
        attrs_set = true;
    }
    if (l.n_chunks > 0) {
        e = timed_launch("chunk_prep", st, [&] {
            chunk_prep_kernel<<<dim3(l.n_chunks, hk_n), kChunkThreads, prep_smem, st>>>(m_qh, m_ql, p);
            return cudaGetLastError();
        });
        if (e != cudaSuccess) return e;
    }
    e = timed_launch("chunk_scan", st, [&] {
        chunk_scan_kernel<<<dim3(hv_n * kSplit, a.n_seq), kChunkThreads, scan_smem, st>>>(
            m_qth, m_qtl, m_wh, m_wl, m_kqh, m_kql, m_kth, m_ktl, p);
        return cudaGetLastError();
    });
    return e;
}

cudaError_t read_device_error(int* code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    }
    return e;
}

}  // namespace gdn
