// Chunked prefill with one decay per key channel (the per-channel decayed
// delta rule that cortiq-engine's pipeline.rs names Mixer::Kda): the per-chunk
// preparation.  The chunk scan is chunk_scan_kda_kernel (gdn_chunked.cu).
//
// With alpha_t = e^{g_t} a vector over the key channels, the token rule
//   S_t = diag(alpha_t) S_{t-1} + beta_t k_t (v_t - (diag(alpha_t) S_{t-1})^T k_t)^T
// unrolled over a chunk that starts from S0, with G_t = sum_{u<=t} g_u (per
// channel, in-chunk), becomes
//   A_ts = beta_t sum_i k_t,i k_s,i e^{G_t,i - G_s,i}  (s < t),  T = (I + A)^-1
//   W = T diag(beta) (K o e^G),   U~ = T diag(beta) V,   U = U~ - W S0
//   O = (Q o e^G) S0 + (M_ts = sum_i q_t,i k_s,i e^{G_t,i - G_s,i}, s <= t) U
//   S1 = diag(e^{G_last}) S0 + (K o e^{G_last - G})^T U
// which is the scalar-decay form with the decay moved inside the key and query
// rows.  The pairwise factors e^{G_t - G_s} cannot be taken outside the
// channel sum, and e^{-G} alone overflows within a chunk, so the Gram matrices
// are formed per 16-token block pair:
//   off the diagonal (s in block b_s < b_t, r = 16 b_t the first token of t's
//   block): e^{G_t - G_s} = e^{G_t - G_r} e^{G_r - G_s}, both factors <= 1, so
//   the block is a product of rescaled key / query rows (warp tensor cores);
//   on the diagonal the factors are taken one pair at a time (CUDA cores).
// One CTA per (chunk, value head) item:
//   tiles   q, k of the key head, v and the gate input a of the value head by TMA
//   G       g = coef softplus(a + dt_bias) from the raw gate input, and its
//           per-channel prefix sums -> shared memory (fp32)
//   rows    K o e^G (operand of W), Q o e^G and K o e^{G_last - G} (workspace,
//           the scan's query rows and state-increment keys), G_last
//   Gram    A and M o QK^T as above; M -> workspace
//   solve   T = (I + A)^-1 (fp32, blocked)
//   [W | U~] = (T diag(beta)) [K o e^G | V] on tcgen05 -> workspace
// Barriers are CTA-wide (__syncthreads) up to the Gram; from the solve to the
// item's end two groups of four warps run apart (named barriers 2 and 3): one
// solves, issues the products and writes W and U~ out, the other forms the
// next item's decays.
#include <algorithm>
#include <atomic>

#include "gdn_chunk_ops.cuh"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
#include "gdn_tma_host.h"

namespace gdn {

using namespace tc;

__device__ int g_kda_error = 0;

__device__ __forceinline__ void report_kda_error(int code) { atomicCAS(&g_kda_error, 0, code); }

constexpr int kKdaThreads = 256;  // 8 warps (more measured slower: register spills, instruction cache)
// shared memory (bytes from a 1024-aligned base); every bf16 tile is 64 rows
// of two 64-column blocks (8 KB each, 128-byte swizzle), hi then lo 16 KB on
constexpr uint32_t kKq = 0;          // Q of the key head
constexpr uint32_t kKk = 32768;      // K of the key head
constexpr uint32_t kKv = 65536;      // V of the value head (MN-major B of U~)
constexpr uint32_t kKg = 98304;      // G, fp32 [64][128] (kda_g)
constexpr uint32_t kKe = 131072;     // K o e^G (MN-major B of W)
constexpr uint32_t kKa = 163840;     // A, fp32 64 x 64 rows (swz_col)
constexpr uint32_t kKt = 180224;     // T, fp32 64 x 64 rows (swz_col)
constexpr uint32_t kKm = 196608;     // M o QK^T staging, bf16 64 x 64 (hi, +8192 lo)
constexpr uint32_t kKb = 212992;     // beta of the chunk's tokens
constexpr uint32_t kKs = 213248;     // first-half channel sums of g, [128] fp32
constexpr uint32_t kKgate = 214016;  // the gate input a of the item, bf16 64 x 128 (TMA, hi only)
constexpr uint32_t kKEnd = 230400;
// T diag(beta), split, is the K-major A operand of [W | U~] (128 rows, 0..63
// written; rows 64..127 read whatever follows): hi over A, lo over the M
// staging, both dead by then.  The Q and K tiles are free once the Gram is
// done, so the next item's land while this one solves.
constexpr uint32_t kKtH = kKa, kKtL = kKm;

// Offset (floats) of G[t][i]: 16-byte chunks XOR-swizzled by 2 (t & 3), so
// that the fragment reads of the block products (rows g and g+8 of a 16-row
// block, two chunks per row) and whole-row reads are free of bank conflicts.
__device__ __forceinline__ int kda_g(int t, int i) {
    return t * kD + ((((i >> 2) ^ ((t & 3) << 1))) << 2) + (i & 3);
}
// Byte offset of element (t, i) in a 64 x 128 bf16 tile.
__device__ __forceinline__ uint32_t kda_el(int t, int i) {
    return (i >> 6) * 8192 + sw128_offset(t, (i & 63) >> 3) + (i & 7) * 2;
}
// Two (hi, lo) elements (t, i), (t, i+1) of a tile as floats.
__device__ __forceinline__ float2 kda_ld2(const uint8_t* tile, uint32_t off) {
    const uint32_t h = *reinterpret_cast<const uint32_t*>(tile + off);
    const uint32_t l = *reinterpret_cast<const uint32_t*>(tile + 16384 + off);
    return make_float2(__uint_as_float(h << 16) + __uint_as_float(l << 16),
                       __uint_as_float(h & 0xFFFF0000u) + __uint_as_float(l & 0xFFFF0000u));
}
// Four (hi, lo) elements (t, i..i+3), i a multiple of 4.
__device__ __forceinline__ void kda_ld4(const uint8_t* tile, uint32_t off, float* f) {
    const uint2 h = *reinterpret_cast<const uint2*>(tile + off);
    const uint2 l = *reinterpret_cast<const uint2*>(tile + 16384 + off);
    f[0] = __uint_as_float(h.x << 16) + __uint_as_float(l.x << 16);
    f[1] = __uint_as_float(h.x & 0xFFFF0000u) + __uint_as_float(l.x & 0xFFFF0000u);
    f[2] = __uint_as_float(h.y << 16) + __uint_as_float(l.y << 16);
    f[3] = __uint_as_float(h.y & 0xFFFF0000u) + __uint_as_float(l.y & 0xFFFF0000u);
}
// One bf16 (hi, lo) element of the M o QK^T staging tile (64 x 64).
__device__ __forceinline__ void kda_st_m(uint8_t* smem, int t, int s, float x) {
    const uint32_t o = sw128_offset(t, s >> 3) + (s & 7) * 2;
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    *reinterpret_cast<__nv_bfloat16*>(smem + kKm + o) = h;
    *reinterpret_cast<__nv_bfloat16*>(smem + kKm + 8192 + o) = __float2bfloat16_rn(x - __bfloat162float(h));
}
// Sum over the warp of each of 32 values, scattered: lane l returns the total
// of v[l] (five halving exchange rounds, 31 shuffles).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool up = (lane & k) != 0;
#pragma unroll
        for (int j = 0; j < k; ++j) {
            const float send = up ? v[j] : v[j + k];
            const float keep = up ? v[j + k] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, k);
        }
    }
    return v[0];
}
// softplus(x) = log(1 + e^x) with the fast exponential and logarithm: log1p
// by Kahan's identity log1p(y) = y log(u) / (u - 1), u = fl(1 + y) (Goldberg,
// "What every computer scientist should know about floating-point arithmetic",
// 1991, theorem 4), which keeps the relative accuracy for small y; the
// identity x above 20, as for the scalar gates.  About 1e-6 relative.
__device__ __forceinline__ float softplus_fast(float x) {
    if (x > 20.f) return x;
    const float y = exp_ftz(x), u = 1.f + y;
    return u == 1.f ? y : log_ftz(u) * (y * rcp_ftz(u - 1.f));
}

// Off-diagonal Gram blocks of key block b_t against n <= 4 8-column tiles cols[j]
// (each in a block b_s < b_t), on one warp: with r = 16 b_t,
//   A_ts += sum_i (k_t,i e^{G_t,i-G_r,i}) (k_s,i e^{G_r,i-G_s,i})
//   M_ts += sum_i (q_t,i e^{G_t,i-G_r,i}) (k_s,i e^{G_r,i-G_s,i})
// as m16n8k16 products of split operands (the row operands formed once for
// all the tiles); A (times beta_t) and M are stored.
constexpr int kKdaTiles = 4;  // column tiles a warp takes at most (n of them used)
__device__ __forceinline__ void kda_gram_offdiag(uint8_t* smem, int bt, const int (&cols)[kKdaTiles], int n, int lane) {
    const float* sG = reinterpret_cast<const float*>(smem + kKg);
    const float* sBeta = reinterpret_cast<const float*>(smem + kKb);
    float* sA = reinterpret_cast<float*>(smem + kKa);
    const int g = lane >> 2, q = lane & 3;
    const int r = 16 * bt, ta = r + g, tb = ta + 8;
    float dA[kKdaTiles][4] = {}, dM[kKdaTiles][4] = {};
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
        const int i0 = 16 * kk + 2 * q, i1 = i0 + 8;
        const float2 gr0 = *reinterpret_cast<const float2*>(sG + kda_g(r, i0));
        const float2 gr1 = *reinterpret_cast<const float2*>(sG + kda_g(r, i1));
        SplitA aq, ak;
        auto left = [&](int t, int i, float2 gr, int slot) {
            const float2 gt = *reinterpret_cast<const float2*>(sG + kda_g(t, i));
            const float e0 = exp_ftz(gt.x - gr.x), e1 = exp_ftz(gt.y - gr.y);
            const uint32_t o = kda_el(t, i);
            const float2 qv = kda_ld2(smem + kKq, o), kv = kda_ld2(smem + kKk, o);
            split2(qv.x * e0, qv.y * e1, aq.h[slot], aq.l[slot]);
            split2(kv.x * e0, kv.y * e1, ak.h[slot], ak.l[slot]);
        };
        left(ta, i0, gr0, 0);
        left(tb, i0, gr0, 1);
        left(ta, i1, gr1, 2);
        left(tb, i1, gr1, 3);
#pragma unroll
        for (int j = 0; j < kKdaTiles; ++j) {
            if (j >= n) break;
            const int s = cols[j] + g;
            const float2 gs0 = *reinterpret_cast<const float2*>(sG + kda_g(s, i0));
            const float2 gs1 = *reinterpret_cast<const float2*>(sG + kda_g(s, i1));
            const float2 k0 = kda_ld2(smem + kKk, kda_el(s, i0)), k1 = kda_ld2(smem + kKk, kda_el(s, i1));
            SplitB b;
            split2(k0.x * exp_ftz(gr0.x - gs0.x), k0.y * exp_ftz(gr0.y - gs0.y), b.h[0], b.l[0]);
            split2(k1.x * exp_ftz(gr1.x - gs1.x), k1.y * exp_ftz(gr1.y - gs1.y), b.h[1], b.l[1]);
            mma16816(dA[j], ak.h, b.h[0], b.h[1]);
            mma16816(dA[j], ak.h, b.l[0], b.l[1]);
            mma16816(dA[j], ak.l, b.h[0], b.h[1]);
            mma16816(dM[j], aq.h, b.h[0], b.h[1]);
            mma16816(dM[j], aq.h, b.l[0], b.l[1]);
            mma16816(dM[j], aq.l, b.h[0], b.h[1]);
        }
    }
    const float ba = sBeta[ta], bb = sBeta[tb];
#pragma unroll
    for (int j = 0; j < kKdaTiles; ++j) {
        if (j >= n) break;
        const int c0 = cols[j] + 2 * q;
        *reinterpret_cast<float2*>(sA + ta * kC + swz_col(ta, c0)) = make_float2(ba * dA[j][0], ba * dA[j][1]);
        *reinterpret_cast<float2*>(sA + tb * kC + swz_col(tb, c0)) = make_float2(bb * dA[j][2], bb * dA[j][3]);
        kda_st_m(smem, ta, c0, dM[j][0]);
        kda_st_m(smem, ta, c0 + 1, dM[j][1]);
        kda_st_m(smem, tb, c0, dM[j][2]);
        kda_st_m(smem, tb, c0 + 1, dM[j][3]);
    }
}

// Diagonal Gram block b: rows ta = 16b + w and tb = 16b + 15 - w (w = 0..7)
// on one warp, whose strictly-lower pairs number w + (15 - w) = 15.  A lane
// takes four channels of every pair, e^{G_t,i - G_s,i} per pair and channel;
// the 15 A and 15 M partial sums and the two diagonal M entries are summed
// over the warp in one scatter, lane l ending with value l.
__device__ __forceinline__ void kda_gram_diag(uint8_t* smem, int b, int w, int lane) {
    const float* sG = reinterpret_cast<const float*>(smem + kKg);
    const float* sBeta = reinterpret_cast<const float*>(smem + kKb);
    float* sA = reinterpret_cast<float*>(smem + kKa);
    const int i4 = 4 * lane;
    auto el4 = [&](int t) { return (uint32_t)((lane >> 4) * 8192) + sw128_offset(t, (lane & 15) >> 1) + (lane & 1) * 8; };
    const int ta = 16 * b + w, tb = 16 * b + 15 - w;
    float ga[4], gb[4], qa[4], qb[4], ka[4], kb[4];
    {
        const float4 x = *reinterpret_cast<const float4*>(sG + kda_g(ta, i4));
        const float4 y = *reinterpret_cast<const float4*>(sG + kda_g(tb, i4));
        ga[0] = x.x; ga[1] = x.y; ga[2] = x.z; ga[3] = x.w;
        gb[0] = y.x; gb[1] = y.y; gb[2] = y.z; gb[3] = y.w;
    }
    kda_ld4(smem + kKq, el4(ta), qa);
    kda_ld4(smem + kKk, el4(ta), ka);
    kda_ld4(smem + kKq, el4(tb), qb);
    kda_ld4(smem + kKk, el4(tb), kb);
    float v[32];
#pragma unroll
    for (int pi = 0; pi < 15; ++pi) {
        const bool ra = pi < w;  // pair (ta, 16b + pi), else (tb, 16b + pi - w)
        const int s = 16 * b + (ra ? pi : pi - w);
        const float4 gs = *reinterpret_cast<const float4*>(sG + kda_g(s, i4));
        float ks[4];
        kda_ld4(smem + kKk, el4(s), ks);
        const float gsv[4] = {gs.x, gs.y, gs.z, gs.w};
        float pa = 0.f, pm = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x = ks[e] * exp_ftz((ra ? ga[e] : gb[e]) - gsv[e]);
            pa = fmaf(ra ? ka[e] : kb[e], x, pa);
            pm = fmaf(ra ? qa[e] : qb[e], x, pm);
        }
        v[pi] = pa;
        v[15 + pi] = pm;
    }
    v[30] = qa[0] * ka[0] + qa[1] * ka[1] + qa[2] * ka[2] + qa[3] * ka[3];
    v[31] = qb[0] * kb[0] + qb[1] * kb[1] + qb[2] * kb[2] + qb[3] * kb[3];
    const float tot = warp_reduce_scatter32(v, lane);
    if (lane < 30) {
        const int pi = lane < 15 ? lane : lane - 15;
        const bool ra = pi < w;
        const int t = ra ? ta : tb, s = 16 * b + (ra ? pi : pi - w);
        if (lane < 15) sA[t * kC + swz_col(t, s)] = sBeta[t] * tot;
        else kda_st_m(smem, t, s, tot);
    } else {
        const int t = lane == 30 ? ta : tb;
        kda_st_m(smem, t, t, tot);
    }
}

// Every thread learns whether any thread passed v != 0 (a CTA barrier).
__device__ __forceinline__ bool kda_any(bool v) { return __syncthreads_or(v ? 1 : 0) != 0; }
// The same over the n threads of named barrier id.
__device__ __forceinline__ bool group_any(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Items blockIdx.x, + gridDim.x, ... of (chunk, value head), chunk-major.
__global__ void __launch_bounds__(kKdaThreads, 1)
chunk_prep_kda_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                      const __grid_constant__ CUtensorMap map_kqh, const __grid_constant__ CUtensorMap map_kql,
                      const __grid_constant__ CUtensorMap map_a, ChunkArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_qk, bar_v, bar_a, bar_mma;
    __shared__ uint32_t tmem_slot;
    float* sG = reinterpret_cast<float*>(smem + kKg);
    float* sBeta = reinterpret_cast<float*>(smem + kKb);
    float* sSum = reinterpret_cast<float*>(smem + kKs);
    float* sA = reinterpret_cast<float*>(smem + kKa);
    float* sT = reinterpret_cast<float*>(smem + kKt);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hv_n = p.n_v_heads, hk_n = p.n_k_heads, R = hv_n / hk_n;
    const int n_items = p.n_chunks * hv_n;

    if (tid == 0) {
        mbar_init(&bar_qk, 1);
        mbar_init(&bar_v, 1);
        mbar_init(&bar_a, 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
        for (const CUtensorMap* m : {&map_qh, &map_ql, &map_kqh, &map_kql, &map_a}) tma_prefetch_desc(m);
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;  // W in columns 0..127, U~ in 128..255
    uint32_t qk_phase = 0, v_phase = 0, a_phase = 0, mma_phase = 0;
    bool qk_pending = false, v_pending = false, a_pending = false, mma_pending = false;

    // q, k tiles of item it's key head; the v tile and the gate input of its
    // value head
    auto issue_qk = [&](int it) {
        const int t0i = p.chunk_info[it / hv_n].x, hk = key_head(it % hv_n, R, hk_n, p.head_map);
        mbar_arrive_expect_tx(&bar_qk, 8 * 8192);
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int col = (m ? hk_n * kD : 0) + hk * kD + 64 * b;
                tma_load_2d(smem + kKq + m * 32768 + b * 8192, &map_qh, &bar_qk, col, t0i);
                tma_load_2d(smem + kKq + m * 32768 + 16384 + b * 8192, &map_ql, &bar_qk, col, t0i);
            }
    };
    auto issue_gate = [&](int it) {
        const int t0i = p.chunk_info[it / hv_n].x;
        mbar_arrive_expect_tx(&bar_a, 2 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b)
            tma_load_2d(smem + kKgate + b * 8192, &map_a, &bar_a, (it % hv_n) * kD + 64 * b, t0i);
    };
    auto issue_v = [&](int it) {
        const int t0i = p.chunk_info[it / hv_n].x, col = 2 * hk_n * kD + (it % hv_n) * kD;
        mbar_arrive_expect_tx(&bar_v, 4 * 8192);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_2d(smem + kKv + b * 8192, &map_qh, &bar_v, col + 64 * b, t0i);
            tma_load_2d(smem + kKv + 16384 + b * 8192, &map_ql, &bar_v, col + 64 * b, t0i);
        }
    };
    if ((int)blockIdx.x < n_items) {
        if (tid == 0) {
            issue_gate(blockIdx.x);
            issue_qk(blockIdx.x);
            issue_v(blockIdx.x);
        }
        qk_pending = v_pending = a_pending = true;
    }
    // rows past the chunk (another sequence's, or padding) of nb 8 KB blocks from base: zero
    auto zero_tail_rows = [&](uint32_t base, int nb, int L) {
        const int nr = kC - L;
        for (int i = tid; i < nr * 8 * nb; i += kKdaThreads) {
            const int ch = i & 7, rest = i >> 3;
            *reinterpret_cast<uint4*>(smem + base + (rest / nr) * 8192 + (L + rest % nr) * 128 + ch * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    };

    // Raw log-decays of item it, g_t,i = coef softplus(a_t,i + dt_bias_i) for
    // t < L (0 past the chunk), from its gate tile into the G tile, by 256
    // threads (j = 0..255: channel j % 128, every other token from j / 128).
    // Formed during the previous item's solve, when the other warps are idle.
    auto raw_g = [&](int it, int j) {
        const int Li = p.chunk_info[it / hv_n].y, hh = it % hv_n, i = j & 127;
        const float A = p.A_log[hh];
        const float coef = p.decay_form ? A : -expf(A), dtb = p.dt_bias[(size_t)hh * kD + i];
        // a rolled loop (straight-line code run once an item is bound by
        // instruction fetch), four loads ahead of their stores
#pragma unroll 1
        for (int k0 = 0; k0 < 32; k0 += 4) {
            float x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                x[k] = __bfloat162float(
                    *reinterpret_cast<const __nv_bfloat16*>(smem + kKgate + kda_el((j >> 7) + 2 * (k0 + k), i)));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = (j >> 7) + 2 * (k0 + k);
                sG[kda_g(t, i)] = t < Li ? coef * softplus_fast(x[k] + dtb) : 0.f;
            }
        }
    };

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int c = item / hv_n, h = item % hv_n;
        const int2 ci = p.chunk_info[c];
        const int t0 = ci.x, L = ci.y;
        const size_t wr = (size_t)item * kC;  // first workspace row of the item
        const int next = item + gridDim.x;
        bool failed = false;
        const int gi = tid & 127, hf = tid >> 7;  // channel, half of the tokens
        const float bt = tid < L ? p.beta[(size_t)(t0 + tid) * hv_n + h] : 0.f;
        do {
            const bool got_qk = mbar_wait(&bar_qk, qk_phase);
            if (kda_any(!got_qk)) {
                if (tid == 0) report_kda_error(13);
                failed = true;
                break;
            }
            qk_pending = false;
            qk_phase ^= 1;
            if (item == (int)blockIdx.x) {  // the first item's raw decays (later ones: during a solve)
                const bool got_a = mbar_wait(&bar_a, a_phase);
                if (kda_any(!got_a)) {
                    if (tid == 0) report_kda_error(13);
                    failed = true;
                    break;
                }
                a_phase ^= 1;
                a_pending = false;
                raw_g(item, tid);
                __syncthreads();
            }
            // the gate tile has been read: the next item's may land now (its
            // raw decays are formed once the Gram has released the G tile)
            if (next < n_items) {
                if (tid == 0) issue_gate(next);
                a_pending = true;
            }
            if (L < kC) zero_tail_rows(kKq, 8, L);
            // G: per-channel prefix sums of the raw decays, the second half of
            // the tokens offset by the first half's sum
            float gv[32];
            {
#pragma unroll
                for (int j = 0; j < 32; ++j) gv[j] = sG[kda_g(32 * hf + j, gi)];
#pragma unroll
                for (int j = 1; j < 32; ++j) gv[j] += gv[j - 1];
                if (hf == 0) sSum[gi] = gv[31];
            }
            if (tid < kC) sBeta[tid] = bt;
            if (tid == 0) bulk_wait_read();  // the last M store has read the staging tile
            __syncthreads();  // (also: every raw value has been read)
            {
                const float off = hf ? sSum[gi] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) sG[kda_g(32 * hf + j, gi)] = gv[j] + off;
            }
            // the M staging tile starts at zero (entries above the diagonal stay so)
            for (int i = tid; i < 1024; i += kKdaThreads)
                *reinterpret_cast<uint4*>(smem + kKm + i * 16) = make_uint4(0u, 0u, 0u, 0u);
            __syncthreads();
            if (tid < kD) p.gcum_ws[(size_t)item * kD + tid] = sG[kda_g(L - 1, tid)];
            // rows: K o e^G (shared memory), Q o e^G and K o e^{G_last - G} (workspace)
            for (int task = tid; task < kC * 16; task += kKdaThreads) {
                const int t = task >> 4, c8 = task & 15;
                float gt[8], gl[8], q8[8], k8[8];
                {
                    const float4 a0 = *reinterpret_cast<const float4*>(sG + kda_g(t, 8 * c8));
                    const float4 a1 = *reinterpret_cast<const float4*>(sG + kda_g(t, 8 * c8 + 4));
                    const float4 l0 = *reinterpret_cast<const float4*>(sG + kda_g(L - 1, 8 * c8));
                    const float4 l1 = *reinterpret_cast<const float4*>(sG + kda_g(L - 1, 8 * c8 + 4));
                    gt[0] = a0.x; gt[1] = a0.y; gt[2] = a0.z; gt[3] = a0.w;
                    gt[4] = a1.x; gt[5] = a1.y; gt[6] = a1.z; gt[7] = a1.w;
                    gl[0] = l0.x; gl[1] = l0.y; gl[2] = l0.z; gl[3] = l0.w;
                    gl[4] = l1.x; gl[5] = l1.y; gl[6] = l1.z; gl[7] = l1.w;
                }
                const uint32_t off = (c8 >> 3) * 8192 + sw128_offset(t, c8 & 7);
                load_pair(smem + kKq + off, smem + kKq + 16384 + off, q8);
                load_pair(smem + kKk + off, smem + kKk + 16384 + off, k8);
                float ke[8], qe[8], kl[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float eg = exp_ftz(gt[e]);
                    ke[e] = k8[e] * eg;
                    qe[e] = q8[e] * eg;
                    kl[e] = k8[e] * exp_ftz(gl[e] - gt[e]);
                }
                split_store(ke, smem + kKe + off, smem + kKe + 16384 + off);
                const size_t qrow = ((size_t)p.qt_row0 + wr + t) * kD + 8 * c8;
                const size_t krow = (wr + t) * kD + 8 * c8;
                split_store(qe, reinterpret_cast<uint8_t*>(p.w_hi + qrow), reinterpret_cast<uint8_t*>(p.w_lo + qrow));
                split_store(kl, reinterpret_cast<uint8_t*>(p.kw_hi + krow), reinterpret_cast<uint8_t*>(p.kw_lo + krow));
            }
            // Gram: the off-diagonal blocks on warps 0..3 (by key block, the
            // 8-column tiles of the blocks before it), then the diagonal blocks
            // on every warp (one row pair of each block)
            if (warp < 4) {
                int cols[kKdaTiles] = {8 * (warp & 1), 16 + 8 * (warp & 1), 32 + 8 * (warp & 1), 0};
                if (warp == 2) cols[0] = 0, cols[1] = 8, cols[2] = 16, cols[3] = 24;
                if (warp == 3) cols[0] = 0, cols[1] = 8;
                kda_gram_offdiag(smem, warp < 2 ? 3 : warp == 2 ? 2 : 1, cols, warp < 2 ? 3 : warp == 2 ? 4 : 2,
                                 lane);
            }
#pragma unroll 1
            for (int b = 0; b < 4; ++b) kda_gram_diag(smem, b, warp, lane);
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tma_store_2d(&map_kqh, smem + kKm, 0, (int)wr);  // M o QK^T rows -> workspace
                tma_store_2d(&map_kql, smem + kKm + 8192, 0, (int)wr);
                bulk_commit();
                if (next < n_items) issue_qk(next);  // the q, k tiles are no longer read
            }
            qk_pending = next < n_items;
            // From here two groups run side by side until the item's end: warps
            // 0, 1, 4, 5 (the accumulator lanes 0..63 are theirs) solve, split T,
            // issue the products and write W and U~ out, on named barriers 2
            // and 3; warps 2, 3, 6, 7 form the next item's raw decays (the G tile
            // is no longer read) once its gate tile, issued at this item's
            // start, has landed.
            bool ok = true;
            if ((warp & 3) < 2) {
                const int w4 = (warp & 1) | ((warp >> 2) << 1), c128 = 32 * w4 + lane;
                solve_unit_lower([&](int r) { return sA + r * kC; }, [&](int r) { return sT + r * kC; }, 2, w4,
                                 lane);
                if (tid == 0) bulk_wait_read();  // the M store has read the staging (T's lo half goes there)
                group_sync(3, 128);
                // T diag(beta), split, as the A tile of the products (blocks
                // above the diagonal are zero; T leaves them unwritten)
                for (int it = c128; it < kC * 8; it += 128) {
                    const int t = it >> 3, ch = it & 7;
                    float f[8];
                    if ((ch >> 1) <= (t >> 4)) {
                        const float4 ta = *reinterpret_cast<const float4*>(sT + t * kC + swz_col(t, 8 * ch));
                        const float4 tb = *reinterpret_cast<const float4*>(sT + t * kC + swz_col(t, 8 * ch + 4));
                        const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = tv[e] * sBeta[8 * ch + e];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = 0.f;
                    }
                    const uint32_t o = sw128_offset(t, ch);
                    split_store(f, smem + kKtH + o, smem + kKtL + o);
                }
                ok = !group_any(3, 128, !mbar_wait(&bar_v, v_phase));  // this item's v tile
                if (ok) {
                    v_pending = false;
                    v_phase ^= 1;
                    if (L < kC) {  // v rows past the chunk: zero
                        const int nr = kC - L;
                        for (int i = c128; i < nr * 8 * 4; i += 128) {
                            const int ch = i & 7, rest = i >> 3;
                            *reinterpret_cast<uint4*>(smem + kKv + (rest / nr) * 8192 + (L + rest % nr) * 128 +
                                                      ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before_sync();
                    group_sync(3, 128);
                    tc_fence_after_sync();
                    if (tid == 0) {  // [W | U~] = (T diag(beta)) [K o e^G | V]
                        const uint32_t th = smem_u32(smem + kKtH), tl = smem_u32(smem + kKtL);
                        const uint32_t ke = smem_u32(smem + kKe), vb = smem_u32(smem + kKv);
                        const uint32_t id = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ah = desc_kmajor_sw128(th + k * 32), al = desc_kmajor_sw128(tl + k * 32);
                            mma3(tmem, ah, al, desc_mnmajor_sw128(ke + k * 2048, 8192),
                                 desc_mnmajor_sw128(ke + 16384 + k * 2048, 8192), id, k > 0 ? 1u : 0u);
                            mma3(tmem + 128, ah, al, desc_mnmajor_sw128(vb + k * 2048, 8192),
                                 desc_mnmajor_sw128(vb + 16384 + k * 2048, 8192), id, k > 0 ? 1u : 0u);
                        }
                        mma_commit(&bar_mma);
                    }
                    mma_pending = true;
                    ok = !group_any(3, 128, !mbar_wait(&bar_mma, mma_phase));
                }
                if (ok) {
                    mma_pending = false;
                    mma_phase ^= 1;
                    tc_fence_after_sync();
                    if (tid == 0 && next < n_items) issue_v(next);  // the products have read the v tile
                    v_pending = next < n_items;
                    // W rows (hi, lo) and U~ rows (fp32, 4-column groups) ->
                    // workspace; warps 4j, 4j+1 take the columns of half j
                    const int qd = warp & 3, half = warp >> 2, t = 32 * qd + lane;
                    const uint32_t lane_base = tmem + ((32u * qd) << 16);
                    float v[64];
                    tmem_ld64(lane_base + 64 * half, v);
                    __nv_bfloat16* wh = p.w_hi + (wr + t) * kD + 64 * half;
                    __nv_bfloat16* wl = p.w_lo + (wr + t) * kD + 64 * half;
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8)
                        split_store(v + 8 * q8, reinterpret_cast<uint8_t*>(wh + 8 * q8),
                                    reinterpret_cast<uint8_t*>(wl + 8 * q8));
                    tmem_ld64(lane_base + 128 + 64 * half, v);
                    float4* dst = reinterpret_cast<float4*>(p.u_ws + wr * kD) + (16 * half) * kC + t;
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4)
                        dst[q4 * kC] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                }
            } else if (next < n_items) {
                const int j0 = 32 * ((warp & 1) | ((warp >> 2) << 1)) + lane;
                ok = mbar_wait(&bar_a, a_phase);
                if (ok) {
                    raw_g(next, j0);
                    raw_g(next, j0 + 128);
                }
            }
            tc_fence_before_sync();
            if (kda_any(!ok)) {
                if (tid == 0) report_kda_error(14);
                failed = true;
                break;
            }
            if (next < n_items) {  // the raw-decay warps took the next item's gate tile
                a_phase ^= 1;
                a_pending = false;
            }
        } while (false);
        if (failed) break;
    }

    // Unwind (also after a give-up): in-flight copies and MMAs land first.
    if (tid == 0) {
        if (qk_pending) mbar_wait(&bar_qk, qk_phase);
        if (a_pending) mbar_wait(&bar_a, a_phase);
        if (v_pending) mbar_wait(&bar_v, v_phase);
    }
    if (kda_any(mma_pending) && tid == 0) mbar_wait(&bar_mma, mma_phase);
    if (tid == 0) bulk_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------- host
size_t kda_prep_smem_bytes() { return 1024 + kKEnd; }

cudaError_t launch_kda_prep(const CUtensorMap& map_qh, const CUtensorMap& map_ql, const CUtensorMap& map_kqh,
                            const CUtensorMap& map_kql, const CUtensorMap& map_a, const ChunkArgs& p, int n_ctas,
                            cudaStream_t st) {
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = kda_prep_smem_bytes();
    if (!attr_set[dev].load()) {
        const cudaError_t e = cudaFuncSetAttribute(chunk_prep_kda_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true);
    }
    chunk_prep_kda_kernel<<<n_ctas, kKdaThreads, smem, st>>>(map_qh, map_ql, map_kqh, map_kql, map_a, p);
    return cudaGetLastError();
}

cudaError_t read_kda_error(int* code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_kda_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_kda_error, &zero, sizeof(int));
    }
    return e;
}

}  // namespace gdn
