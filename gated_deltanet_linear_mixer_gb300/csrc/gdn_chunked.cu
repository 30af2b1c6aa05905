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
//   chunk_scan  one CTA per (sequence, value head): carries S in fp32
//               registers across the chunks; per chunk three MMA groups
//               ([W; e^G Q] S,  then (M o QK^T) U and (e^{G_last-G} K)^T U),
//               the state update and the fused gated RMSNorm epilogue.
// Every operand tile is either loaded by TMA with the 128-byte swizzle or
// written by threads in the same layout; operands whose contraction runs
// along a tile's rows use the MN-major descriptor, so no tile is ever
// transposed.
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
constexpr uint32_t kPrepSmemFixed = 81920;   // Ag 32K + T 16K + B 32K
constexpr uint32_t kScanSmem = 131072;       // Bs 32K + Aw 32K + Aq 16K + Bu 16K + Ak 16K + Ut 16K

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

// --------------------------------------------------------------- chunk_prep
__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_prep_kernel(const __grid_constant__ CUtensorMap map_qkv, ChunkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sAg = smem;            // [Q; K] K-major, 2 column blocks of 128 rows x 128 B
    uint8_t* sT = smem + 32768;     // T, K-major 128 rows (64..127 zero) x 128 B
    uint8_t* sB = smem + 49152;     // [beta e^G K | beta V], MN-major 64 rows x 256
    const int R = p.n_v_heads / p.n_k_heads;
    float* sAt = reinterpret_cast<float*>(smem + kPrepSmemFixed);  // per head A^T [s][t]
    float* sG = sAt + R * kC * kC;
    float* sBeta = sG + R * kC;
    __shared__ __align__(8) uint64_t bar_tma, bar_mma;
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
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    for (int i = tid; i < 512; i += kChunkThreads)
        reinterpret_cast<uint4*>(sT + 8192)[i] = make_uint4(0u, 0u, 0u, 0u);
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
    const uint32_t tmem = tmem_slot;
    uint32_t mma_phase = 0;
    bool tma_issued = false, mma_pending = false;

    do {
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_tma, 4 * 8192);
            const int qc = hk * kD, kc = p.n_k_heads * kD + hk * kD;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tma_load_2d(sAg + b * 16384, &map_qkv, &bar_tma, qc + 64 * b, t0);
                tma_load_2d(sAg + b * 16384 + 8192, &map_qkv, &bar_tma, kc + 64 * b, t0);
            }
        }
        tma_issued = true;
        if (any_failed(mbar_wait(&bar_tma, 0))) {
            if (tid == 0) report_error(1);
            break;
        }
        tma_issued = false;
        if (L < kC) {  // rows past the chunk belong to another sequence: zero them
            const int nr = kC - L;
            for (int i = tid; i < nr * 32; i += kChunkThreads) {
                const int ch = i & 7, rest = i >> 3;
                const int r = L + rest % nr, pb = rest / nr;  // pb: part (q/k) x block
                *reinterpret_cast<uint4*>(sAg + (pb >> 1) * 16384 + ((pb & 1) * 64 + r) * 128 +
                                          ch * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (tid == 0) {  // Gram: rows 0..63 = Q K^T, rows 64..127 = K K^T
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t a = smem_u32(sAg) + (k >> 2) * 16384 + (k & 3) * 32;
                mma_bf16(tmem, desc_kmajor_sw128(a), desc_kmajor_sw128(a + 8192),
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
        if (warp < 4) {
            float v[64];
            tmem_ld32(tmem + ((32u * warp) << 16), v);
            tmem_ld32(tmem + ((32u * warp) << 16) + 32, v + 32);
            if (warp < 2) {  // masked decayed Q K^T rows -> workspace
                const int t = 32 * warp + lane;
                for (int r = 0; r < R; ++r) {
                    const float Gt = sG[r * kC + t];
                    uint4* dst = reinterpret_cast<uint4*>(
                        p.qk_ws + ((size_t)(c * hv_n + hk * R + r) * kC + t) * kC);
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int s = q8 * 8 + e;
                            f[e] = s <= t ? expf(Gt - sG[r * kC + s]) * v[s] : 0.f;
                        }
                        dst[q8] = pack_bf16x8(f);
                    }
                }
            } else {  // A = strictly-lower beta_t e^{G_t-G_s} k_t.k_s, stored transposed
                const int t = 32 * (warp - 2) + lane;
                for (int r = 0; r < R; ++r) {
                    const float Gt = sG[r * kC + t], bt = sBeta[r * kC + t];
                    float* At = sAt + r * kC * kC;
#pragma unroll
                    for (int s = 0; s < kC; ++s)
                        At[s * kC + t] = s < t ? bt * expf(Gt - sG[r * kC + s]) * v[s] : 0.f;
                }
            }
        }
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();

        bool failed = false;
        for (int r = 0; r < R && !failed; ++r) {
            const int h = hk * R + r;
            if (warp < 2) {
                // T = (I + A)^-1: thread j solves (I + A) x = e_j by forward
                // substitution, eliminating one known entry at a time.
                const int j = tid;
                const float* At = sAt + r * kC * kC;
                float x[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) x[t] = t == j ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < kC - 1; ++s) {
                    const float xs = x[s];
#pragma unroll
                    for (int t = s + 1; t < kC; ++t) x[t] = fmaf(-At[s * kC + t], xs, x[t]);
                }
#pragma unroll
                for (int t = 0; t < kC; ++t)
                    *reinterpret_cast<__nv_bfloat16*>(sT + t * 128 + ((((j >> 3) ^ (t & 7))) << 4) +
                                                      (j & 7) * 2) = __float2bfloat16_rn(x[t]);
            } else if (warp >= 4) {
                // B rows s: [beta_s e^{G_s} k_s | beta_s v_s], MN-major
                for (int it = tid - 128; it < kC * 32; it += 128) {
                    const int ch = it & 7, blk = (it >> 3) & 3, s = it >> 5;
                    const uint32_t pos = static_cast<uint32_t>((ch ^ (s & 7)) << 4);
                    const float bt = sBeta[r * kC + s];
                    uint4 val = make_uint4(0u, 0u, 0u, 0u);
                    if (blk < 2) {
                        const uint4 src =
                            *reinterpret_cast<const uint4*>(sAg + blk * 16384 + (64 + s) * 128 + pos);
                        val = scale_bf16x8(src, bt * expf(sG[r * kC + s]));
                    } else if (s < L) {
                        const uint4 src = *reinterpret_cast<const uint4*>(
                            p.qkv + (size_t)(t0 + s) * cd + 2 * p.n_k_heads * kD + h * kD +
                            (blk - 2) * 64 + ch * 8);
                        val = scale_bf16x8(src, bt);
                    }
                    *reinterpret_cast<uint4*>(sB + blk * 8192 + s * 128 + pos) = val;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
            if (tid == 0) {  // [W | U~] = T [beta e^G K | beta V]   (M padded to 128)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sT) + k * 32),
                             desc_mnmajor_sw128(smem_u32(sB) + k * 2048, 8192),
                             idesc_bf16_f32(128, 256, false, true), k > 0 ? 1u : 0u);
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
            if ((warp & 3) < 2) {  // rows t of W (warps 0,1) and of U~ (warps 4,5)
                const int t = 32 * (warp & 3) + lane;
                const int col0 = (warp >> 2) * 128;
                __nv_bfloat16* dst =
                    (warp < 4 ? p.w_ws : p.u_ws) + ((size_t)(c * hv_n + h) * kC + t) * kD;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    float v[32];
                    tmem_ld32(tmem + ((32u * (warp & 3)) << 16) + col0 + 32 * cb, v);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        reinterpret_cast<uint4*>(dst + 32 * cb)[q8] = pack_bf16x8(v + 8 * q8);
                }
            }
            if (tid < kC) p.gcum_ws[(size_t)(c * hv_n + h) * kC + tid] = sG[r * kC + tid];
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
        }
    } while (false);

    // Unwind after a give-up: let in-flight copies and MMAs land first.
    if (tma_issued) mbar_wait(&bar_tma, 0);
    if (mma_pending) mbar_wait(&bar_mma, mma_phase);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// --------------------------------------------------------------- chunk_scan
__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_u, const __grid_constant__ CUtensorMap map_qk,
                  ChunkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sBs = smem;            // S (bf16), MN-major: 128 key rows x 128 value lanes
    uint8_t* sAw = smem + 32768;    // [W; e^G Q] K-major, 2 column blocks x 128 rows
    uint8_t* sAq = smem + 65536;    // [0; M o QK^T] K-major, 128 rows x 64
    uint8_t* sBu = smem + 81920;    // U (bf16), MN-major: 64 token rows x 128 value lanes
    uint8_t* sAk = smem + 98304;    // e^{G_last-G} K, MN-major: 64 token rows x 128 key lanes
    uint8_t* sUt = smem + 114688;   // U~ rows (K-major, 2 column blocks x 64 rows)
    __shared__ float sG[kC];
    __shared__ float sSsq[2][kC];
    __shared__ __align__(8) uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hf = warp >> 2;
    const int row = 32 * q + lane;  // tensor-memory lane this thread reads
    const int h = blockIdx.x, n = blockIdx.y;
    const int hv_n = p.n_v_heads;
    const int R = hv_n / p.n_k_heads, hk = h / R;
    const int bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    const int c_begin = p.cu_chunks[n], c_end = p.cu_chunks[n + 1];
    const size_t slab = ((size_t)n * hv_n + h) * kD * kD;

    // fp32 state: this thread owns S[row][64*hf .. 64*hf+63]
    float S[64];
    if (p.state_in) {
        const float4* src = reinterpret_cast<const float4*>(p.state_in + slab + (size_t)row * kD + 64 * hf);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 v = src[i];
            S[4 * i] = v.x; S[4 * i + 1] = v.y; S[4 * i + 2] = v.z; S[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) S[i] = 0.f;
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(sBs + hf * 16384 + row * 128 + ((ch ^ (row & 7)) << 4)) =
            pack_bf16x8(S + 8 * ch);
    for (int i = tid; i < 512; i += kChunkThreads)
        reinterpret_cast<uint4*>(sAq)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;               // cols 0..127: [W S; Q S + (M o QK^T) U]
    const uint32_t tmem_s = tmem + 128;            // cols 128..255: K'^T U
    const uint32_t lane_off = (32u * q) << 16;
    uint32_t ld_phase = 0, mma_phase = 0;
    bool ld_pending = false, mma_pending = false;
    const bool act_is_sigmoid = p.act == 1;

    for (int c = c_begin; c < c_end; ++c) {
        const int t0 = bos + (c - c_begin) * kC;
        const int L = min(kC, eos - t0);
        const int wrow = (c * hv_n + h) * kC;
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_ld, 8 * 8192 + 8192);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tma_load_2d(sAw + b * 16384, &map_w, &bar_ld, 64 * b, wrow);
                tma_load_2d(sAw + b * 16384 + 8192, &map_qkv, &bar_ld, hk * kD + 64 * b, t0);
                tma_load_2d(sAk + b * 8192, &map_qkv, &bar_ld,
                            p.n_k_heads * kD + hk * kD + 64 * b, t0);
                tma_load_2d(sUt + b * 8192, &map_u, &bar_ld, 64 * b, wrow);
            }
            tma_load_2d(sAq + 8192, &map_qk, &bar_ld, 0, wrow);
        }
        ld_pending = true;
        if (tid < kC) sG[tid] = p.gcum_ws[(size_t)wrow + tid];
        if (any_failed(mbar_wait(&bar_ld, ld_phase))) {
            if (tid == 0) report_error(4);
            break;
        }
        ld_pending = false;
        ld_phase ^= 1;
        const float GL = sG[L - 1];
        // Scale Q rows by e^{G_t} and K rows by e^{G_last-G_s}; zero rows >= L.
        for (int it = tid; it < 2048; it += kChunkThreads) {
            const int ch = it & 7, b = (it >> 3) & 1, r = (it >> 4) & 63, which = it >> 10;
            uint8_t* ptr = which == 0 ? sAw + b * 16384 + (64 + r) * 128 + ch * 16
                                      : sAk + b * 8192 + r * 128 + ch * 16;
            const float f = r < L ? expf(which == 0 ? sG[r] : GL - sG[r]) : 0.f;
            *reinterpret_cast<uint4*>(ptr) = scale_bf16x8(*reinterpret_cast<const uint4*>(ptr), f);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (tid == 0) {  // [W S ; e^G Q S]
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sAw) + (k >> 2) * 16384 + (k & 3) * 32),
                         desc_mnmajor_sw128(smem_u32(sBs) + k * 2048, 16384),
                         idesc_bf16_f32(128, 128, false, true), k > 0 ? 1u : 0u);
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        if (any_failed(mbar_wait(&bar_mma, mma_phase))) {
            if (tid == 0) report_error(5);
            break;
        }
        mma_pending = false;
        mma_phase ^= 1;
        tc_fence_after_sync();
        if (q < 2) {  // U = U~ - W S for token row `row`, value lanes of half hf
            float u[64];
            tmem_ld32(tmem + lane_off + 64 * hf, u);
            tmem_ld32(tmem + lane_off + 64 * hf + 32, u + 32);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint32_t pos = static_cast<uint32_t>((ch ^ (row & 7)) << 4);
                float ut[8];
                unpack_bf16x8(*reinterpret_cast<const uint4*>(sUt + hf * 8192 + row * 128 + pos), ut);
#pragma unroll
                for (int e = 0; e < 8; ++e) ut[e] -= u[8 * ch + e];
                *reinterpret_cast<uint4*>(sBu + hf * 8192 + row * 128 + pos) = pack_bf16x8(ut);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (tid == 0) {
            // O rows: e^G Q S + (M o QK^T) U  (rows 0..63 of A are zero)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sAq) + k * 32),
                         desc_mnmajor_sw128(smem_u32(sBu) + k * 2048, 8192),
                         idesc_bf16_f32(128, 128, false, true), 1u);
            // state increment: (e^{G_last-G} K)^T U
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem_s, desc_mnmajor_sw128(smem_u32(sAk) + k * 2048, 8192),
                         desc_mnmajor_sw128(smem_u32(sBu) + k * 2048, 8192),
                         idesc_bf16_f32(128, 128, true, true), k > 0 ? 1u : 0u);
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        if (any_failed(mbar_wait(&bar_mma, mma_phase))) {
            if (tid == 0) report_error(6);
            break;
        }
        mma_pending = false;
        mma_phase ^= 1;
        tc_fence_after_sync();
        {  // S <- e^{G_last} S + K'^T U ; refresh the bf16 copy
            const float gam = expf(GL);
            float ds[64];
            tmem_ld32(tmem_s + lane_off + 64 * hf, ds);
            tmem_ld32(tmem_s + lane_off + 64 * hf + 32, ds + 32);
#pragma unroll
            for (int j = 0; j < 64; ++j) S[j] = fmaf(gam, S[j], ds[j]);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(sBs + hf * 16384 + row * 128 + ((ch ^ (row & 7)) << 4)) =
                    pack_bf16x8(S + 8 * ch);
        }
        if (q >= 2) {  // output rows: partial sum of squares over this half
            float o[64];
            tmem_ld32(tmem + lane_off + 64 * hf, o);
            tmem_ld32(tmem + lane_off + 64 * hf + 32, o + 32);
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) ss = fmaf(o[j], o[j], ss);
            sSsq[hf][row - 64] = ss;
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (q >= 2) {  // gated RMSNorm epilogue for token t
            const int t = row - 64;
            if (t < L) {
                float o[64];
                tmem_ld32(tmem + lane_off + 64 * hf, o);
                tmem_ld32(tmem + lane_off + 64 * hf + 32, o + 32);
                const float rr = rsqrtf((sSsq[0][t] + sSsq[1][t]) * (1.f / kD) + p.rms_eps);
                const size_t base = (size_t)(t0 + t) * hv_n * kD + (size_t)h * kD + 64 * hf;
                const uint4* zp = reinterpret_cast<const uint4*>(p.z + base);
                uint4* op = reinterpret_cast<uint4*>(p.out + base);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float zz[8], y[8];
                    unpack_bf16x8(zp[ch], zz);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float gate = act_is_sigmoid ? sigmoidf_(zz[e]) : siluf_(zz[e]);
                        y[e] = o[8 * ch + e] * rr * p.norm_w[64 * hf + 8 * ch + e] * gate;
                    }
                    op[ch] = pack_bf16x8(y);
                }
            }
            tc_fence_before_sync();
        }
    }

    if (ld_pending) mbar_wait(&bar_ld, ld_phase);
    if (mma_pending) mbar_wait(&bar_mma, mma_phase);
    if (p.state_out) {
        float4* dst = reinterpret_cast<float4*>(p.state_out + slab + (size_t)row * kD + 64 * hf);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------- host
size_t chunked_workspace_bytes(int n_seq, const int32_t* cu_host, int n_k_heads, int n_v_heads,
                               ChunkLayout* lay) {
    ChunkLayout l{};
    const int T = n_seq > 0 ? cu_host[n_seq] : 0;
    long long chunks = 0;
    for (int i = 0; i < n_seq; ++i) chunks += (cu_host[i + 1] - cu_host[i] + kC - 1) / kC;
    const size_t cd = 2 * (size_t)n_k_heads * kD + (size_t)n_v_heads * kD;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    size_t off = 0;
    l.qkv = off; off = up(off + (size_t)T * cd * 2);
    l.g = off; off = up(off + (size_t)T * n_v_heads * 4);
    l.beta = off; off = up(off + (size_t)T * n_v_heads * 4);
    l.cu_chunks = off; off = up(off + (size_t)(n_seq + 1) * 4);
    l.w = off; off = up(off + (size_t)chunks * n_v_heads * kC * kD * 2);
    l.u = off; off = up(off + (size_t)chunks * n_v_heads * kC * kD * 2);
    l.qk = off; off = up(off + (size_t)chunks * n_v_heads * kC * kC * 2);
    l.gcum = off; off = up(off + (size_t)chunks * n_v_heads * kC * 4);
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

    // 1. prologue: conv + SiLU + L2 norm + gates -> qkv, g, beta (workspace)
    ConvArgs cv{};
    cv.n_seq = a.n_seq; cv.n_tokens = T; cv.n_k_heads = hk_n; cv.n_v_heads = hv_n;
    cv.d_k = kD; cv.d_v = kD; cv.conv_k = a.conv_k; cv.l2_eps = a.l2_eps;
    cv.cu_seqlens = a.cu_seqlens; cv.x = a.x; cv.a = a.a; cv.b = a.b;
    cv.conv_w = a.conv_w; cv.A_log = a.A_log; cv.dt_bias = a.dt_bias;
    cv.conv_state_in = a.conv_state_in;
    cv.qkv_out = ws + l.qkv;
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
    p.qkv = reinterpret_cast<const __nv_bfloat16*>(ws + l.qkv);
    p.g = reinterpret_cast<const float*>(ws + l.g);
    p.beta = reinterpret_cast<const float*>(ws + l.beta);
    p.z = static_cast<const __nv_bfloat16*>(a.z);
    p.norm_w = a.norm_w;
    p.state_in = a.state_in; p.state_out = a.state_out;
    p.w_ws = reinterpret_cast<__nv_bfloat16*>(ws + l.w);
    p.u_ws = reinterpret_cast<__nv_bfloat16*>(ws + l.u);
    p.qk_ws = reinterpret_cast<__nv_bfloat16*>(ws + l.qk);
    p.gcum_ws = reinterpret_cast<float*>(ws + l.gcum);
    p.out = static_cast<__nv_bfloat16*>(a.out);

    // Tensor maps; with no chunk at all (only empty sequences) no kernel
    // dereferences them and they stay zero.
    CUtensorMap m_qkv, m_w, m_u, m_qk;
    std::memset(&m_qkv, 0, sizeof(m_qkv));
    m_w = m_u = m_qk = m_qkv;
    const uint64_t wrows = (uint64_t)l.n_chunks * hv_n * kC;
    if (l.n_chunks > 0) {
        if (!make_tma_map_bf16_2d(&m_qkv, ws + l.qkv, T, cd, cd, 64, 64) ||
            !make_tma_map_bf16_2d(&m_w, ws + l.w, wrows, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_u, ws + l.u, wrows, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_qk, ws + l.qk, wrows, kC, kC, 64, 64))
            return cudaErrorInvalidValue;
    }

    const size_t prep_smem = 1024 + kPrepSmemFixed + (size_t)R * (kC * kC * 4 + 2 * kC * 4);
    const size_t scan_smem = 1024 + kScanSmem;
    static bool attrs_set = false;
    if (!attrs_set) {
        cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             1024 + kPrepSmemFixed + 4 * (kC * kC * 4 + 2 * kC * 4));
        cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(scan_smem));
        attrs_set = true;
    }
    if (l.n_chunks > 0) {
        e = timed_launch("chunk_prep", st, [&] {
            chunk_prep_kernel<<<dim3(l.n_chunks, hk_n), kChunkThreads, prep_smem, st>>>(m_qkv, p);
            return cudaGetLastError();
        });
        if (e != cudaSuccess) return e;
    }
    e = timed_launch("chunk_scan", st, [&] {
        chunk_scan_kernel<<<dim3(hv_n, a.n_seq), kChunkThreads, scan_smem, st>>>(m_qkv, m_w, m_u,
                                                                                m_qk, p);
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
