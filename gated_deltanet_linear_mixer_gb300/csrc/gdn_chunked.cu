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
//   chunk_fused both phases in one launch (prep CTAs publish each item's
//               flag; scan clusters wait on it), for batches whose scan alone
//               would leave most SMs idle; the two-kernel form serves the rest.
// Every operand tile is either loaded by TMA with the 128-byte swizzle or
// written by threads in the same layout.  B operands whose contraction runs
// along a tile's rows (S, U, [K|V] rows) use the MN-major descriptor; every A
// operand is K-major (the one A that would be MN-major, the scaled keys of the
// state increment, is transposed by threads).
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_chunk_ops.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma_host.h"

namespace gdn {

using namespace tc;

constexpr int kChunkThreads = 256;

__device__ int g_device_error = 0;

__device__ __forceinline__ void report_error(int code) { atomicCAS(&g_device_error, 0, code); }

// --------------------------------------------------------------- chunk_prep
// One CTA per (chunk, key head); its R = Hv/Hk value heads are processed in
// pairs so that every phase keeps all eight warps busy: the two heads of a
// pair occupy rows 0..63 and 64..127 of each M=128 product.
//   Gram     [Q; K] K^T on the tensor core (shared by the heads); the K tile
//            itself -> workspace, rows in chunk order (the scan's K^T U')
//   per pair: M o QK^T rows -> workspace; A = strictly-lower beta_t
//            e^{G_t-G_s} k_t.k_s; T = (I + A)^-1 by a blocked solve in fp32;
//            W = (T diag(beta e^G)) K and U~ = (T diag(beta)) V on the tensor
//            core (the row scalings of the right-hand sides are folded into
//            T's columns); everything -> workspace.
constexpr uint32_t kPrepAg = 0;          // [Q; K] K-major 128 x 128 (hi at +0, lo at +32768)
constexpr uint32_t kPrepV = 65536;       // V of the pair: hi blocks (a0 a1 b0 b1) then lo blocks
constexpr uint32_t kPrepT1 = 131072;     // [T'_a; T'_b] K-major 128 x 64 (hi, lo at +16384)
constexpr uint32_t kPrepT2 = 163840;     // [T''_a; T''_b]
constexpr uint32_t kPrepVec = 196608;    // G, beta per value head
// tensor-memory columns
constexpr uint32_t kTpW = 0, kTpUa = 128, kTpUb = 256, kTpGram = 384;

// fp32 T of head hh (0/1) of the pair: rows live in the shared memory of the
// (then dead) Q rows of the Gram operand, 32 rows per 8 KB piece.
__device__ __forceinline__ float* prep_tf(uint8_t* smem, int hh, int row) {
    return reinterpret_cast<float*>(smem + kPrepAg + (hh * 2 + (row >> 5)) * 16384 + (row & 31) * 256);
}

// Items worker, worker + n_workers, ... (chunk-major).
__device__ __forceinline__ void chunk_prep_body(const CUtensorMap& map_qh, const CUtensorMap& map_ql,
                                                const CUtensorMap& map_wh, const CUtensorMap& map_wl,
                                                const CUtensorMap& map_kqh,
                                                const CUtensorMap& map_kql, const CUtensorMap& map_kwh,
                                                const CUtensorMap& map_kwl, const ChunkArgs& p,
                                                const int worker, const int n_workers) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int R = p.n_v_heads / p.n_k_heads;
    float* sG = reinterpret_cast<float*>(smem + kPrepVec);
    float* sBeta = sG + R * kC;
    float* sCs1 = sBeta + R * kC;  // beta_s e^{G_s}: column factors of T'
    float* sCs2 = sCs1 + R * kC;   // beta_s: column factors of T''
    __shared__ __align__(8) uint64_t bar_tma, bar_mma, bar_v;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hv_n = p.n_v_heads;
    const int n_pairs = (R + 1) / 2;
    const int n_items = p.n_chunks * p.n_k_heads;  // (chunk, key head), chunk-major

    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_v, 1);
        fence_barrier_init();
        for (const CUtensorMap* m : {&map_qh, &map_ql, &map_wh, &map_wl, &map_kqh, &map_kql, &map_kwh, &map_kwl})
            tma_prefetch_desc(m);
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 512);
    tc_fence_before_sync();
    prep_sync();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    uint32_t mma_phase = 0, tma_phase = 0, v_phase = 0;
    bool tma_pending = false, mma_pending = false, v_pending = false;

    // q rows (0..63) and k rows (64..127) of item it, both column blocks
    auto issue_qk_tiles = [&](int it, int t0i) {  // t0i: first token of item it's chunk
        const int hki = it % p.n_k_heads;
        mbar_arrive_expect_tx(&bar_tma, 8 * 8192);
        const int qc = hki * kD, kc = p.n_k_heads * kD + hki * kD;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            tma_load_2d(smem + kPrepAg + b * 16384, &map_qh, &bar_tma, qc + 64 * b, t0i);
            tma_load_2d(smem + kPrepAg + b * 16384 + 8192, &map_qh, &bar_tma, kc + 64 * b, t0i);
            tma_load_2d(smem + kPrepAg + 32768 + b * 16384, &map_ql, &bar_tma, qc + 64 * b, t0i);
            tma_load_2d(smem + kPrepAg + 32768 + b * 16384 + 8192, &map_ql, &bar_tma, kc + 64 * b, t0i);
        }
    };
    // v rows of pair pr of item it: hi blocks at kPrepV + (2*slot + b) * 8192,
    // lo blocks 32 KB further
    auto issue_v_item = [&](int it, int t0i, int pr) {
        const int hki = it % p.n_k_heads;
        const int nb = min(2, R - 2 * pr);
        mbar_arrive_expect_tx(&bar_v, nb * 4 * 8192);
        for (int sl = 0; sl < nb; ++sl) {
            const int vc = 2 * p.n_k_heads * kD + value_head(hki, 2 * pr + sl, R, p.n_k_heads, p.head_map) * kD;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tma_load_2d(smem + kPrepV + (2 * sl + b) * 8192, &map_qh, &bar_v, vc + 64 * b, t0i);
                tma_load_2d(smem + kPrepV + 32768 + (2 * sl + b) * 8192, &map_ql, &bar_v, vc + 64 * b, t0i);
            }
        }
    };
    // Chunk position (first token, length) of an item two items ahead, and the
    // gate inputs of the next item (whose position is then in hand): neither
    // load waits on the other.
    auto info = [&](int it) { return it < n_items ? p.chunk_info[it / p.n_k_heads] : make_int2(0, 0); };
    int2 ci_n = make_int2(0, 0);                   // the next item's (at the top of an item)
    int2 ci_nn = info(worker + n_workers);          // the one after
    float ng0 = 0.f, ng1 = 0.f, nb0 = 0.f, nb1 = 0.f;
    auto prefetch_gates = [&](int it) {  // ci_n holds item it's position
        if (warp < R) {
            const int h = value_head(it % p.n_k_heads, warp, R, p.n_k_heads, p.head_map);
            const int s0 = 2 * lane, s1 = 2 * lane + 1;
            ng0 = ng1 = nb0 = nb1 = 0.f;
            if (s0 < ci_n.y) {
                ng0 = p.g[(size_t)(ci_n.x + s0) * hv_n + h];
                nb0 = p.beta[(size_t)(ci_n.x + s0) * hv_n + h];
            }
            if (s1 < ci_n.y) {
                ng1 = p.g[(size_t)(ci_n.x + s1) * hv_n + h];
                nb1 = p.beta[(size_t)(ci_n.x + s1) * hv_n + h];
            }
        }
    };
    if (worker < n_items) {
        ci_n = info(worker);
        prefetch_gates(worker);
        if (tid == 0) {
            issue_qk_tiles(worker, ci_n.x);
            issue_v_item(worker, ci_n.x, 0);
        }
    }
    tma_pending = v_pending = worker < n_items;
    int pub = -1;  // finished item whose flag is still to be set

    for (int item = worker; item < n_items; item += n_workers) {
    const int c = item / p.n_k_heads, hk = item % p.n_k_heads;
    const int next = item + n_workers;
    const int t0 = ci_n.x, L = ci_n.y;
    bool failed = false;
    const float g0 = ng0, g1 = ng1, b0 = nb0, b1 = nb1;
    ci_n = ci_nn;                              // the next item's position, loaded an item ago
    ci_nn = info(next + n_workers);
    if (next < n_items) prefetch_gates(next);  // lands while this item runs
    if (warp < R) {  // cumulative log-decay and write strength of value head hk*R + warp
        const int s0 = 2 * lane, s1 = 2 * lane + 1;
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
        sCs1[warp * kC + s0] = b0 * exp_ftz(excl + g0);
        sCs1[warp * kC + s1] = b1 * exp_ftz(excl + g0 + g1);
        sCs2[warp * kC + s0] = b0;
        sCs2[warp * kC + s1] = b1;
    }
    do {
        if (prep_failed(mbar_wait(&bar_tma, tma_phase))) {  // this item's q, k tiles
            if (tid == 0) report_error(1);
            failed = true;
            break;
        }
        tma_pending = false;
        tma_phase ^= 1;
        if (L < kC) {  // rows past the chunk belong to another sequence: zero them
            const int nr = kC - L;
            for (int i = tid; i < nr * 64; i += kChunkThreads) {
                const int ch = i & 7, rest = i >> 3;
                const int r = L + rest % nr, pb = rest / nr;  // pb: hi/lo x part x block
                *reinterpret_cast<uint4*>(smem + kPrepAg + (pb >> 2) * 32768 + ((pb >> 1) & 1) * 16384 +
                                          ((pb & 1) * 64 + r) * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        prep_sync();
        tc_fence_after_sync();
        if (tid == 0) {  // Gram: rows 0..63 = Q K^T, rows 64..127 = K K^T
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                const uint32_t ah = smem_u32(smem + kPrepAg) + off, al = ah + 32768;
                mma3(tmem + kTpGram, desc_kmajor_sw128(ah), desc_kmajor_sw128(al),
                     desc_kmajor_sw128(ah + 8192), desc_kmajor_sw128(al + 8192),
                     idesc_bf16_f32(128, 64), k > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma);
            const int krow = (c * p.n_k_heads + hk) * kC;  // K tile (rows past the chunk are 0)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tma_store_2d(&map_kwh, smem + kPrepAg + b * 16384 + 8192, 64 * b, krow);
                tma_store_2d(&map_kwl, smem + kPrepAg + 32768 + b * 16384 + 8192, 64 * b, krow);
            }
            bulk_commit();
        }
        mma_pending = true;
        if (prep_failed(mbar_wait(&bar_mma, mma_phase))) {
            if (tid == 0) report_error(2);
            failed = true;
            break;
        }
        mma_pending = false;
        mma_phase ^= 1;
        tc_fence_after_sync();
        if (pub >= 0) {  // the previous item's stores were issued long ago
            if (tid == 0) publish_item(p.ready + pub);
            pub = -1;
        }

        for (int pr = 0; pr < n_pairs; ++pr) {
            const int nb = min(2, R - 2 * pr);
            if (prep_failed(mbar_wait(&bar_v, v_phase))) {  // this pair's v tiles
                if (tid == 0) report_error(7);
                failed = true;
                break;
            }
            v_pending = false;
            v_phase ^= 1;
            if (L < kC) {  // v rows past the chunk: zero (they may hold anything)
                const int nr = kC - L;
                for (int i = tid; i < nr * 64; i += kChunkThreads) {
                    const int ch = i & 7, rest = i >> 3;
                    const int r = L + rest % nr, blk = rest / nr;  // blk: hi/lo x slot x block
                    *reinterpret_cast<uint4*>(smem + kPrepV + blk * 8192 + r * 128 + ch * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (tid == 0) bulk_wait_read();  // the last W stores have read T1 / T2
            prep_sync();
            // ---- phase A: M o QK^T rows (warps 0,1 / 4,5) and A^T (warps 2,3 / 6,7)
            {
                const int hh = warp >> 2;             // head of the pair this warp serves
                const int q = warp & 3;
                const int t = 32 * (q & 1) + lane;    // token row
                float v[64];
                tmem_ld64(tmem + kTpGram + ((32u * q) << 16), v);
                if (hh < nb) {
                    const int r = 2 * pr + hh, h = value_head(hk, r, R, p.n_k_heads, p.head_map);
                    const float* Gr = sG + r * kC;
                    const float Gt = Gr[t];
                    if (q < 2) {  // masked decayed Q K^T row t -> staging tile (hi, lo)
                        uint8_t* st = smem + kPrepT2 + hh * 16384;
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8) {
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int s = q8 * 8 + e;
                                f[e] = s <= t ? exp_ftz(Gt - Gr[s]) * v[s] : 0.f;
                            }
                            const uint32_t o = sw128_offset(t, q8);
                            split_store(f, st + o, st + 8192 + o);
                        }
                        (void)h;
                    } else {  // A[t][s] = beta_t e^{G_t-G_s} k_t.k_s for s < t, row t, swizzled
                        float* sA = reinterpret_cast<float*>(smem + kPrepT1 + hh * 16384) + t * kC;
                        const float bt = sBeta[r * kC + t];
#pragma unroll
                        for (int c4 = 0; c4 < 16; ++c4) {
                            float f[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int s = 4 * c4 + e;
                                f[e] = s < t ? bt * exp_ftz(Gt - Gr[s]) * v[s] : 0.f;
                            }
                            *reinterpret_cast<float4*>(sA + ((c4 ^ (t & 15)) << 2)) =
                                make_float4(f[0], f[1], f[2], f[3]);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            prep_sync();
            if (tid == 64) {  // M o QK^T tiles -> workspace (thread 64 idles in the diagonal solve)
                for (int hh = 0; hh < nb; ++hh) {
                    const int row = (c * hv_n + value_head(hk, 2 * pr + hh, R, p.n_k_heads, p.head_map)) * kC;
                    tma_store_2d(&map_kqh, smem + kPrepT2 + hh * 16384, 0, row);
                    tma_store_2d(&map_kql, smem + kPrepT2 + hh * 16384 + 8192, 0, row);
                }
                bulk_commit();
            }
            // ---- phase B: T = (I + A)^-1 per head (four warps a head)
            {
                const int hh = warp >> 2;
                if (hh < nb) {
                    float* sAf = reinterpret_cast<float*>(smem + kPrepT1 + hh * 16384);
                    solve_unit_lower([&](int r) { return sAf + r * kC; },
                                     [&](int r) { return prep_tf(smem, hh, r); }, 2 + hh, warp & 3, lane);
                }
            }
            if (tid == 64) bulk_wait_all();  // the QK^T tiles have landed (T2 is rewritten next)
            prep_sync();
            // ---- T' = T diag(beta e^G), T'' = T diag(beta): split into the A tiles
            for (int it = tid; it < 2 * kC * 8; it += kChunkThreads) {
                const int hh = it >> 9, t = (it >> 3) & 63, ch = it & 7;
                float f1[8], f2[8];
                // blocks above the diagonal are zero (never written by the solve)
                if (hh < nb && (ch >> 1) <= (t >> 4)) {
                    const int r = 2 * pr + hh;
                    const float* tr = prep_tf(smem, hh, t);
                    const float4 ta = *reinterpret_cast<const float4*>(tr + swz_col(t, 8 * ch));
                    const float4 tb = *reinterpret_cast<const float4*>(tr + swz_col(t, 8 * ch + 4));
                    const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = 8 * ch + e;
                        f1[e] = tv[e] * sCs1[r * kC + s];
                        f2[e] = tv[e] * sCs2[r * kC + s];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f1[e] = f2[e] = 0.f;
                }
                const int row = 64 * hh + t;
                const uint32_t o = row * 128 + ((ch ^ (row & 7)) << 4);
                split_store(f1, smem + kPrepT1 + o, smem + kPrepT1 + 16384 + o);
                split_store(f2, smem + kPrepT2 + o, smem + kPrepT2 + 16384 + o);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            prep_sync();
            tc_fence_after_sync();
            // ---- phase C: W = [T'_a; T'_b] K ; U~_x = [T''_a; T''_b] V_x
            if (tid == 0) {
                const uint32_t t1 = smem_u32(smem + kPrepT1), t2 = smem_u32(smem + kPrepT2);
                const uint32_t kb = smem_u32(smem + kPrepAg) + 8192;   // K rows, MN-major B
                const uint32_t vb = smem_u32(smem + kPrepV);
                const uint32_t id = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma3(tmem + kTpW, desc_kmajor_sw128(t1 + k * 32), desc_kmajor_sw128(t1 + 16384 + k * 32),
                         desc_mnmajor_sw128(kb + k * 2048, 16384), desc_mnmajor_sw128(kb + 32768 + k * 2048, 16384),
                         id, k > 0 ? 1u : 0u);
                for (int sl = 0; sl < nb; ++sl) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma3(tmem + (sl ? kTpUb : kTpUa), desc_kmajor_sw128(t2 + k * 32),
                             desc_kmajor_sw128(t2 + 16384 + k * 32),
                             desc_mnmajor_sw128(vb + sl * 16384 + k * 2048, 8192),
                             desc_mnmajor_sw128(vb + 32768 + sl * 16384 + k * 2048, 8192), id,
                             k > 0 ? 1u : 0u);
                }
                mma_commit(&bar_mma);
            }
            mma_pending = true;
            if (prep_failed(mbar_wait(&bar_mma, mma_phase))) {
                if (tid == 0) report_error(3);
                failed = true;
                break;
            }
            mma_pending = false;
            mma_phase ^= 1;
            tc_fence_after_sync();
            if (pr + 1 == n_pairs && next < n_items) {
                // the q, k tiles are no longer read (the products are
                // done): the next item's may land while this one is written out
                if (tid == 0) {
                    bulk_wait_read();  // the K tile store has read the tile
                    issue_qk_tiles(next, ci_n.x);
                }
                tma_pending = true;
            }
            if (tid == 0) {  // the products have read the v tiles: the next ones may land
                if (pr + 1 < n_pairs) issue_v_item(item, t0, pr + 1);
                else if (next < n_items) issue_v_item(next, ci_n.x, 0);
            }
            v_pending = pr + 1 < n_pairs || next < n_items;
            // ---- phase D: W rows (hi, lo) staged in the free T tiles (head a in
            // T1, head b in T2) for TMA stores; U~ rows (fp32) straight to the
            // workspace, 4-column groups of 64 rows each ([group][row][4]), so
            // that both these stores and the scan's row loads are coalesced
            {
                const int q = warp & 3, half = warp >> 2;
                const int hh = q >> 1, t = 32 * (q & 1) + lane;
                uint8_t* st = smem + (hh ? kPrepT2 : kPrepT1);
                float v[64];
                tmem_ld64(tmem + kTpW + ((32u * q) << 16) + 64 * half, v);
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const uint32_t o = half * 8192 + sw128_offset(t, q8);
                    split_store(v + 8 * q8, st + o, st + 16384 + o);
                }
                tmem_ld64(tmem + (hh ? kTpUb : kTpUa) + ((32u * q) << 16) + 64 * half, v);
                if (hh < nb) {
                    const int h = value_head(hk, 2 * pr + hh, R, p.n_k_heads, p.head_map);
                    float4* dst = reinterpret_cast<float4*>(p.u_ws + (size_t)(c * hv_n + h) * kC * kD) +
                                  (16 * half) * kC + t;
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4)
                        dst[q4 * kC] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                    if (half == 0) p.gcum_ws[(size_t)(c * hv_n + h) * kC + t] = sG[(2 * pr + hh) * kC + t];
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            prep_sync();
            tc_fence_after_sync();
            if (tid == 0) {
                for (int hh = 0; hh < nb; ++hh) {
                    const int row = (c * hv_n + value_head(hk, 2 * pr + hh, R, p.n_k_heads, p.head_map)) * kC;
                    const uint8_t* st = smem + (hh ? kPrepT2 : kPrepT1);
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        tma_store_2d(&map_wh, st + b * 8192, 64 * b, row);
                        tma_store_2d(&map_wl, st + 16384 + b * 8192, 64 * b, row);
                    }
                }
                bulk_commit();  // waited (reads) before T1 / T2 are next written
            }
            prep_sync();
        }
        if (!failed && p.ready) {
            if (item == worker) {
                // a CTA's first item is published as soon as its stores have
                // landed: the first chunk rows gate the scan's start, while later
                // rows are ready long before the scan reaches them
                if (tid == 0) publish_item(p.ready + item);
            } else {
                pub = item;  // published after the next item's Gram, when its stores are long done
            }
        }
    } while (false);
    if (failed) break;
    }

    // Unwind (also after a give-up): in-flight copies and MMAs land first.
    if (tid == 0) {
        if (tma_pending) mbar_wait(&bar_tma, tma_phase);
        if (v_pending) mbar_wait(&bar_v, v_phase);
    }
    if (prep_any(mma_pending) && tid == 0) mbar_wait(&bar_mma, mma_phase);
    if (tid == 0) bulk_wait_all();
    if (tid == 0 && pub >= 0) publish_item(p.ready + pub);
    tc_fence_before_sync();
    prep_sync();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void __launch_bounds__(kChunkThreads, 1)
chunk_prep_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                  const __grid_constant__ CUtensorMap map_wh, const __grid_constant__ CUtensorMap map_wl,
                  const __grid_constant__ CUtensorMap map_kqh, const __grid_constant__ CUtensorMap map_kql,
                  const __grid_constant__ CUtensorMap map_kwh, const __grid_constant__ CUtensorMap map_kwl,
                  ChunkArgs p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the scan may start in our tail
    chunk_prep_body(map_qh, map_ql, map_wh, map_wl, map_kqh, map_kql, map_kwh, map_kwl, p,
                    blockIdx.x, gridDim.x);
}

// --------------------------------------------------------------- chunk_scan
// A cluster of kSplit CTAs shares one (sequence, value head): CTA p owns value
// lanes [64p, 64p+64) of the state, of U and of the outputs.  The state
// recurrence per chunk is a chain of two tensor-core products,
//   U = U~ - W S   (rows 0..63 of P4 = [W; Q] S),   S <- e^{G_last} S + K''^T U
// (P7, K'' = diag(e^{G_last-G}) K, formed as K^T U' with U' = diag(e^{G_last-G})
// U, so that the key tile is chunk_prep's copy of its input and the decay
// factors, all <= 1, scale the fp32 U before it is split).
//
// Warp roles (12 warps launched at 168 registers a thread; a register split
// gives the eight compute warps 200 and the control warpgroup 96: 256 x 200 +
// 128 x 96 = 63,488, within the launch's 384 x 168 = 64,512; 176 and 120 in
// the per-channel decay instance):
//   warps 0..7  compute.  Thread (warp w, lane l) owns key lane 32 (w%4) + l
//               of the state and value lanes 32 (w/4) .. +31 of this CTA's
//               slice, which is exactly the part of the tensor-memory
//               accumulators that the warp may read.  Warps 0,1,4,5
//               (accumulator rows 0..63) form U_c; warps 2,3,6,7 (rows
//               64..127) write the output of chunk c-1,
//               o = e^{G_t} (Q S)_t + ((M o QK^T) U)_t with the gated RMSNorm
//               (sums of squares exchanged with the peer CTA through
//               distributed shared memory), reading their accumulators before
//               their share of the state update and finishing after it; all
//               eight update the state.
//   warp 8      one lane issues the chain's MMAs: P4_c, then, once U'_c is in
//               shared memory, P7_c.
//   warp 9      one lane issues every TMA and bulk copy, each as soon as the
//               readers of the buffer's previous contents are done (and, in the
//               fused launch, the chunk's prep rows are published), and the
//               output term P6_c = (M o QK^T)_c U_c once P7_c is done, so that
//               it runs in the pipe while the state is updated.
//   warps 10,11 the gate norm_w act(z) of each chunk, from its z rows, into
//               shared memory for the output warps.
// Split products: every product is hi.hi + hi.lo + lo.hi.  In the fused
// launch P4 takes the hi and lo halves of its B operand side by side as one
// N=128 product, A_hi [B_hi | B_lo], plus A_lo B_hi into the first half, its
// result the sum of the accumulator's two halves; in the two-kernel launch,
// and for P7 and P6 in both, the three terms are N=64 MMAs into one
// accumulator, so that a reader takes one 32-column block.  Every wait is
// bounded (wait_or_dead).
constexpr int kSplit = 2;
constexpr int kDS = kD / kSplit;      // value lanes per CTA
constexpr int kScanThreads = 384;     // 8 compute warps + a control warpgroup
constexpr int kComputeThreads = 256;
// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t kScanBsH = 0, kScanBsL = 16384;          // S, MN-major 128 x 64 (lo = 2nd N block)
constexpr uint32_t kScanA4H = 32768, kScanA4L = 65536;      // [W; Q] K-major 128 x 128 (hi, lo)
constexpr uint32_t kScanKH = 98304, kScanKL = 114688;       // K as MN-major A (dk 128 x t 64)
constexpr uint32_t kScanBu = 131072;                        // U, MN-major 64 x 64 (hi, +8192 lo)
constexpr uint32_t kScanQk = 147456;                        // M o QK^T rows, K-major 64 x 64 (hi, +8192 lo)
constexpr uint32_t kScanUp = 163840;                        // U' = diag(e^{G_last-G}) U (hi, +8192 lo)
constexpr uint32_t kScanGate = 180224;                      // norm_w act(z), fp32 64 x 64 (rows 256 B,
                                                            //   16-byte chunks swizzled by the row)
constexpr uint32_t kScanUt = 196608;                        // U~ of the chunk, fp32 [16 groups][64][4]
constexpr uint32_t kScanZ = 212992;                         // z rows, bf16 64 x 64 (TMA, 128-byte swizzle)
constexpr uint32_t kScanGc = 221184;                        // in-chunk cumulative log-decay, 2 x 64 fp32
constexpr uint32_t kScanEnd = 221696;
constexpr uint32_t kScanGl = kScanEnd;                      // per-channel decay: G_last per key
                                                            //   channel, 2 x 128 fp32
constexpr uint32_t kScanEndKda = kScanGl + 2 * 128 * 4;
// tensor-memory columns: P4 in two slots (chunk c uses c%2) of 128 columns (64
// in the two-kernel launch), P7 in 64 columns, P6 in two 64-column slots
constexpr uint32_t kTmD4 = 0, kTmDs = 256, kTmD6 = 320;

struct ScanSync {
    uint64_t a4, k, qk;        // TMA loads landed
    uint64_t s_lo, s_hi;       // S_c rows 0..63 / 64..127 split into shared memory (128 threads each)
    uint64_t p4, p7, p6[2];    // MMA groups done (tcgen05.commit)
    uint64_t u, u2;            // U'_c, then U_c, in shared memory (128 U threads)
    uint64_t d4free[2];        // output warps have read slot c%2 of P4 and P6 (128 threads)
    uint64_t gate;             // the gate warps have written the gate (64 threads)
    uint64_t ug, zf;           // U~ and G of a chunk, its z rows, landed (bulk copies)
    uint64_t x[2], xf[2];      // peer's sums of squares arrived / slot free
    int dead;
    int n_a4, n_k, n_qk, n_ug, n_zf;  // copies issued per barrier (producer)
    int n_commits;             // MMA groups committed (issuer)
    uint32_t last_commit;      // barrier index and parity of the issuer's last commit
    int n_p6;                  // P6 groups committed (producer)
};

// Bounded wait that also gives up as soon as another thread of this CTA (or,
// with peer_dead != 0, of the peer CTA) has recorded a failure; the failure
// and timeout checks run every 16th round.
__device__ __forceinline__ bool wait_or_dead(uint64_t* bar, uint32_t parity, ScanSync& sy,
                                             int code, bool cluster_scope = false,
                                             uint32_t peer_dead = 0) {
    auto tryw = [&] {
        return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (tryw()) return true;
    const uint64_t t0 = globaltimer_ns();
    const long long c0 = clock64();
    for (uint32_t it = 0;; ++it) {
        if (tryw()) return true;
        if ((it & 15u) != 15u) continue;
        if (*reinterpret_cast<volatile int*>(&sy.dead)) return false;
        if (peer_dead && ld_cluster_s32(peer_dead)) {
            atomicExch(&sy.dead, 1);
            return false;
        }
        if (globaltimer_ns() - t0 > 2000000000ull || clock64() - c0 > (1ll << 32)) {
            atomicExch(&sy.dead, 1);
            report_error(code);
            return false;
        }
    }
}

// Value head h of sequence n, this CTA's half of the value lanes.  kSplitP4:
// P4 as three N=64 products into one 64-column accumulator from a rolled issue
// loop, instead of the N-stacked form.  The two-kernel scan takes it: with the
// scan on every SM at once, its shorter U step and smaller hot code (the
// instruction cache) measured faster.  The fused launch keeps the stacked
// form, where eight fewer MMAs on the chain count for more; the two launches
// therefore differ in that product's rounding.
// kKda: one decay per key channel.  The query rows of P4 are chunk_prep_kda's
// Q o e^G (per value head, from the W arrays at row qt_row0 on), the keys of
// P7 its K o e^{G_last - G} (per value head), so U' = U and the output takes
// no e^{G_t} factor; the state decays by e^{G_last} per key row.
template <bool kSplitP4, bool kKda>
__device__ __forceinline__ void chunk_scan_body(const CUtensorMap& map_qh, const CUtensorMap& map_ql,
                                                const CUtensorMap& map_wh, const CUtensorMap& map_wl,
                                                const CUtensorMap& map_kqh, const CUtensorMap& map_kql,
                                                const CUtensorMap& map_kwh, const CUtensorMap& map_kwl,
                                                const CUtensorMap& map_z, const ChunkArgs& p, const int h,
                                                const int n) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ ScanSync sy;
    __shared__ float sx[2][kC];   // the peer's per-token sums of squares
    __shared__ float sSq[2][kC];  // this CTA's, per 32-lane half
    __shared__ float sNw[kDS];    // this CTA's norm weights
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int v0 = static_cast<int>(rank) * kDS;  // first value lane of this CTA
    const int hv_n = p.n_v_heads;
    const int R = hv_n / p.n_k_heads, hk = key_head(h, R, p.n_k_heads, p.head_map);
    const int bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
    const int c_begin = p.cu_chunks[n], n_ch = p.cu_chunks[n + 1] - c_begin;
    const size_t slab = ((size_t)n * hv_n + h) * kD * kD;
    const int qcol = hk * kD;

    if (tid < kDS) sNw[tid] = p.norm_w[v0 + tid];
    if (tid == 0) {
        mbar_init(&sy.a4, 1);
        mbar_init(&sy.k, 1); mbar_init(&sy.qk, 1);
        mbar_init(&sy.s_lo, 128); mbar_init(&sy.s_hi, 128);
        mbar_init(&sy.p4, 1); mbar_init(&sy.p7, 1);
        mbar_init(&sy.p6[0], 1); mbar_init(&sy.p6[1], 1);
        mbar_init(&sy.u, 128); mbar_init(&sy.u2, 128);
        mbar_init(&sy.d4free[0], 128); mbar_init(&sy.d4free[1], 128);
        mbar_init(&sy.gate, 64);
        mbar_init(&sy.ug, 1); mbar_init(&sy.zf, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sy.x[i], 1);
            mbar_init(&sy.xf[i], 64);
        }
        sy.dead = 0;
        sy.n_a4 = sy.n_k = sy.n_qk = sy.n_ug = sy.n_zf = 0;
        sy.n_commits = 0;
        sy.n_p6 = 0;
        sy.last_commit = 0;
        fence_barrier_init();
        for (const CUtensorMap* m : {&map_qh, &map_ql, &map_wh, &map_wl, &map_kqh, &map_kql, &map_kwh, &map_kwl, &map_z})
            tma_prefetch_desc(m);
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 512);
    tc_fence_before_sync();
    cluster_arrive();  // the peer's barriers are initialised before any remote arrive
    cluster_wait();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    constexpr uint32_t kP4Cols = kSplitP4 ? 64 : 128;  // tensor-memory columns of a P4 slot
    const uint32_t peer_dead = map_to_rank(smem_u32(&sy.dead), peer);

    auto wrow = [&](int c) { return ((c_begin + c) * hv_n + h) * kC; };
    auto tok0 = [&](int c) { return bos + c * kC; };
    auto chunk_len = [&](int c) { return min(kC, eos - tok0(c)); };
    // Fused launch: chunk c's workspace rows come from prep CTAs running
    // alongside; the calling thread waits (bounded) for its item flag with a
    // gpu-scope acquire before it reads them.  TMA loads of published rows
    // follow a global proxy fence (in the issue_* helpers).
    auto wait_chunk = [&](int c) -> bool {
        if (!p.ready || c >= n_ch) return true;
        const int* f = p.stall_flag ? p.stall_flag : p.ready + (size_t)(c_begin + c) * p.n_k_heads + hk;
        if (ld_acquire_gpu(f)) return true;
        const uint64_t t0 = globaltimer_ns();
        const long long c0 = clock64();
        for (;;) {
            __nanosleep(100);
            if (ld_acquire_gpu(f)) return true;
            if (*reinterpret_cast<volatile int*>(&sy.dead)) return false;
            if (globaltimer_ns() - t0 > p.wait_ns || clock64() - c0 > (1ll << 32)) {
                atomicExch(&sy.dead, 1);
                report_error(11);
                return false;
            }
        }
    };

    if (warp >= 8) {
        // ------------------------------------------------ control warpgroup
        // per-channel decay: 120 / 176 (its control code needs more; spills
        // measured 6% slower at 96 / 200); 128 x 120 + 256 x 176 = 60,416
        regs_dec<kKda ? 120 : 96>();
        if (warp == 8 && lane == 0 && n_ch > 0) {
            // MMA issuer.  Shared-memory descriptors, computed once: a
            // descriptor for address a + o is the one for a plus o >> 4 (the
            // 14-bit start field cannot carry over, every address here is below
            // 256 KB).
            const uint64_t dA4 = desc_kmajor_sw128(smem_u32(smem + kScanA4H));
            const uint64_t dBs = desc_mnmajor_sw128(smem_u32(smem + kScanBsH), 16384);
            const uint64_t dK = desc_mnmajor_sw128(smem_u32(smem + kScanKH), 8192);
            const uint64_t dUp = desc_mnmajor_sw128(smem_u32(smem + kScanUp), 8192);
            constexpr uint64_t kLo16 = 16384 >> 4, kLoA4 = 32768 >> 4;
            const uint32_t id128 = idesc_bf16_f32(128, 2 * kDS, false, true);
            const uint32_t id64 = idesc_bf16_f32(128, kDS, false, true);
            const uint32_t id7_64 = idesc_bf16_f32(128, kDS, true, true);
            uint32_t last = 0;  // (barrier index << 1) | parity of the last commit
            int commits = 0;
            for (int c = 0; c < n_ch; ++c) {
                // P4_c = [W; Q] S_c into slot c%2: A_hi [S_hi | S_lo] + A_lo S_hi,
                // the key lanes 0..63 as soon as the warps owning those state rows
                // have stored them, then 64..127
                if (!wait_or_dead(&sy.a4, c & 1, sy, 4) || !wait_or_dead(&sy.s_lo, c & 1, sy, 4))
                    break;
                // slot c%2 last held chunk c-2, whose output must have been read
                // from it (the state rows 0..63 do not imply that)
                if (c >= 2 && !wait_or_dead(&sy.d4free[c & 1], ((c - 2) >> 1) & 1, sy, 4)) break;
                tc_fence_after_sync();
                const uint32_t d4 = tmem + kTmD4 + (uint32_t)(c & 1) * kP4Cols;
                bool hi_ok = true;
                if constexpr (kSplitP4) {
#pragma unroll 1
                    for (int k = 0; k < 8; ++k) {
                        if (k == 4) {
                            if (!(hi_ok = wait_or_dead(&sy.s_hi, c & 1, sy, 4))) break;
                            tc_fence_after_sync();
                        }
                        const uint64_t ao = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                        mma3(d4, dA4 + ao, dA4 + kLoA4 + ao, dBs + k * 128, dBs + kLo16 + k * 128, id64,
                             k > 0 ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (k == 4) {
                            if (!(hi_ok = wait_or_dead(&sy.s_hi, c & 1, sy, 4))) break;
                            tc_fence_after_sync();
                        }
                        const uint64_t ao = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
                        mma_bf16(d4, dA4 + ao, dBs + k * 128, id128, k > 0 ? 1u : 0u);
                        mma_bf16(d4, dA4 + kLoA4 + ao, dBs + k * 128, id64, 1u);
                    }
                }
                if (!hi_ok) {  // the MMAs already issued still complete before the unwind
                    mma_commit(&sy.p4);
                    last = (0u << 1) | (c & 1); ++commits;
                    break;
                }
                mma_commit(&sy.p4);
                last = (0u << 1) | (c & 1); ++commits;
                // P7_c = K^T U'_c, three N=64 products into one accumulator
                if (!wait_or_dead(&sy.u, c & 1, sy, 6) || !wait_or_dead(&sy.k, c & 1, sy, 5)) break;
                tc_fence_after_sync();
#pragma unroll 1  // few registers: the control warps run at 96
                for (int k = 0; k < 4; ++k) {
                    mma3(tmem + kTmDs, dK + k * 128, dK + kLo16 + k * 128, dUp + k * 128,
                         dUp + (8192 >> 4) + k * 128, id7_64, k > 0 ? 1u : 0u);
                }
                mma_commit(&sy.p7);
                last = (1u << 1) | (c & 1); ++commits;
            }
            sy.n_commits = commits;
            sy.last_commit = last;
        } else if (warp >= 10 && n_ch > 0) {
            // gate warps: norm_w act(z) of token row t = 32 (warp - 10) + lane of
            // each chunk, from its z rows, once the output warps have read the
            // previous chunk's gate
            const int t = 32 * (warp - 10) + lane;
            const bool sigmoid_gate = p.act == 1;
            float* gb = reinterpret_cast<float*>(smem + kScanGate) + t * kC;
            const uint8_t* zrow = smem + kScanZ + t * 128;
            for (int c = 0; c < n_ch; ++c) {
                if (!wait_or_dead(&sy.zf, c & 1, sy, 12) ||
                    (c > 0 && !wait_or_dead(&sy.d4free[(c - 1) & 1], ((c - 1) >> 1) & 1, sy, 9)))
                    break;
#pragma unroll 2
                for (int i = 0; i < 8; ++i) {  // 16-byte chunk i of the z row: value lanes 8i .. 8i+7
                    float zz[8], gv[8];
                    unpack_bf16x8(*reinterpret_cast<const uint4*>(zrow + ((i ^ (t & 7)) << 4)), zz);
                    if (sigmoid_gate) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) gv[e] = sNw[8 * i + e] * sigmoidf_(zz[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) gv[e] = sNw[8 * i + e] * siluf_(zz[e]);
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2)
                        *reinterpret_cast<float4*>(gb + (((2 * i + h2) ^ (t & 15)) << 2)) =
                            make_float4(gv[4 * h2], gv[4 * h2 + 1], gv[4 * h2 + 2], gv[4 * h2 + 3]);
                }
                mbar_arrive(&sy.gate);  // also releases the z buffer
            }
        } else if (warp == 9 && lane == 0 && n_ch > 0) {
            // TMA producer
            auto issue_a4 = [&](int c) {  // W rows (0..63) and q rows (64..127), both column blocks
                if (p.ready) fence_proxy_async_global();
                mbar_arrive_expect_tx(&sy.a4, 8 * 8192);
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    tma_load_2d(smem + kScanA4H + b * 16384, &map_wh, &sy.a4, 64 * b, wrow(c));
                    tma_load_2d(smem + kScanA4L + b * 16384, &map_wl, &sy.a4, 64 * b, wrow(c));
                    if constexpr (kKda) {
                        tma_load_2d(smem + kScanA4H + b * 16384 + 8192, &map_wh, &sy.a4, 64 * b, p.qt_row0 + wrow(c));
                        tma_load_2d(smem + kScanA4L + b * 16384 + 8192, &map_wl, &sy.a4, 64 * b, p.qt_row0 + wrow(c));
                    } else {
                        tma_load_2d(smem + kScanA4H + b * 16384 + 8192, &map_qh, &sy.a4, qcol + 64 * b, tok0(c));
                        tma_load_2d(smem + kScanA4L + b * 16384 + 8192, &map_ql, &sy.a4, qcol + 64 * b, tok0(c));
                    }
                }
                sy.n_a4 += 1;
            };
            auto issue_k = [&](int c) {  // key rows of the chunk, both key-lane blocks (MN-major A)
                if (p.ready) fence_proxy_async_global();
                const int krow = kKda ? wrow(c) : ((c_begin + c) * p.n_k_heads + hk) * kC;
                mbar_arrive_expect_tx(&sy.k, 4 * 8192);
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    tma_load_2d(smem + kScanKH + b * 8192, &map_kwh, &sy.k, 64 * b, krow);
                    tma_load_2d(smem + kScanKL + b * 8192, &map_kwl, &sy.k, 64 * b, krow);
                }
                sy.n_k += 1;
            };
            auto issue_qk = [&](int c) {  // masked decayed Q K^T rows
                if (p.ready) fence_proxy_async_global();
                mbar_arrive_expect_tx(&sy.qk, 2 * 8192);
                tma_load_2d(smem + kScanQk, &map_kqh, &sy.qk, 0, wrow(c));
                tma_load_2d(smem + kScanQk + 8192, &map_kql, &sy.qk, 0, wrow(c));
                sy.n_qk += 1;
            };
            // the chunk's U~ rows (this CTA's 64 value lanes: 16 contiguous
            // 4-column groups) and its cumulative log-decay, into G buffer c%2
            auto issue_ug = [&](int c) {
                if (p.ready) fence_proxy_async_global();
                mbar_arrive_expect_tx(&sy.ug, 16384 + (kKda ? kD : kC) * 4);
                bulk_load_1d(smem + kScanUt, p.u_ws + (size_t)wrow(c) * kD + (size_t)(v0 >> 2) * kC * 4,
                             16384, &sy.ug);
                if constexpr (kKda)
                    bulk_load_1d(smem + kScanGl + (c & 1) * kD * 4,
                                 p.gcum_ws + (size_t)((c_begin + c) * hv_n + h) * kD, kD * 4, &sy.ug);
                else
                    bulk_load_1d(smem + kScanGc + (c & 1) * kC * 4, p.gcum_ws + wrow(c), kC * 4, &sy.ug);
                sy.n_ug += 1;
            };
            auto issue_z = [&](int c) {  // the chunk's z rows, this CTA's value lanes
                mbar_arrive_expect_tx(&sy.zf, 8192);
                tma_load_2d(smem + kScanZ, &map_z, &sy.zf, h * kD + v0, tok0(c));
                sy.n_zf += 1;
            };
            // P6_c = (M o QK^T)_c U_c into slot c%2, once U_c is in shared memory and
            // P7_c is done (P6 then runs while the state is updated).  A rows
            // 0..63 of this M=128 operand are whatever precedes the QK^T rows in
            // shared memory: they only reach accumulator rows 0..63, which
            // nothing reads.
            const uint64_t dBu = desc_mnmajor_sw128(smem_u32(smem + kScanBu), 8192);
            const uint64_t dQk = desc_kmajor_sw128(smem_u32(smem + kScanQk) - 8192);
            constexpr uint64_t kLo8 = 8192 >> 4;
            const uint32_t id64 = idesc_bf16_f32(128, kDS, false, true);
            auto issue_p6 = [&](int c) -> bool {
                if (!wait_or_dead(&sy.u2, c & 1, sy, 6) || !wait_or_dead(&sy.qk, c & 1, sy, 8)) return false;
                tc_fence_after_sync();
#pragma unroll 1  // few registers: the control warps run at 96 (off the chain)
                for (int k = 0; k < 4; ++k)
                    mma3(tmem + kTmD6 + (uint32_t)(c & 1) * 64, dQk + k * 2, dQk + kLo8 + k * 2,
                         dBu + k * 128, dBu + kLo8 + k * 128, id64, k > 0 ? 1u : 0u);
                mma_commit(&sy.p6[c & 1]);
                sy.n_p6 += 1;
                return true;
            };
            // Two-kernel launch of the scalar form: this scan is the prep's
            // programmatic dependent and may start in the prep's tail; its
            // first copy of prep rows waits for the prep grid's completion (and
            // its writes).  Nothing else this CTA reads before then is written
            // by the prep.  (Without a pending prerequisite the wait returns at
            // once: the per-channel scan is launched after its prep.)
            if (!p.ready) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                fence_proxy_async_global();  // the rows are read by TMA (the async proxy)
            }
            bool ok = wait_chunk(0);
            if (ok) {
                issue_ug(0);
                issue_z(0);
                issue_a4(0);
                issue_k(0);
                issue_qk(0);
            }
            for (int c = 0; ok && c + 1 < n_ch; ++c) {
                if (!(ok = wait_chunk(c + 1))) break;
                // [W; Q]_{c+1} once P4_c has read [W; Q]_c
                if (!(ok = wait_or_dead(&sy.p4, c & 1, sy, 5))) break;
                issue_a4(c + 1);
                // U~_{c+1} once the U warps have read U~_c, G_{c+1} into the buffer
                // the output warps read chunk c-1's from before arriving on d4free
                if (!(ok = wait_or_dead(&sy.u, c & 1, sy, 6) &&
                           (c == 0 || wait_or_dead(&sy.d4free[(c - 1) & 1], ((c - 1) >> 1) & 1, sy, 7))))
                    break;
                issue_ug(c + 1);
                // K_{c+1} once P7_c has read K_c
                if (!(ok = wait_or_dead(&sy.p7, c & 1, sy, 5))) break;
                issue_k(c + 1);
                if (!(ok = issue_p6(c))) break;
                // z_{c+1} once the gate warps have turned z_c into the gate
                if (!(ok = wait_or_dead(&sy.gate, c & 1, sy, 9))) break;
                issue_z(c + 1);
                // QK^T_{c+1} once P6_c has read QK^T_c
                if (!(ok = wait_or_dead(&sy.p6[c & 1], (c >> 1) & 1, sy, 7))) break;
                issue_qk(c + 1);
            }
            // the last chunk's output term, after its P7
            if (ok && wait_or_dead(&sy.p7, (n_ch - 1) & 1, sy, 5)) issue_p6(n_ch - 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ compute warps
        regs_inc<kKda ? 176 : 200>();
        const int q = warp & 3, half = warp >> 2;
        const int row = 32 * q + lane;       // accumulator lane: key lane / token row
        const int cl = 32 * half;            // first of this thread's 32 value lanes in the slice
        const uint32_t lane_off = (32u * q) << 16;
        const bool is_u = q < 2;  // warps 0,1,4,5: accumulator rows 0..63

        float S[32];  // S[row][v0 + cl .. +31]
        if (p.state_in) {
            const float4* src = reinterpret_cast<const float4*>(p.state_in + slab + (size_t)row * kD + v0 + cl);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = src[i];
                S[4 * i] = v.x; S[4 * i + 1] = v.y; S[4 * i + 2] = v.z; S[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) S[i] = 0.f;
        }
        auto store_s = [&] {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint32_t o = row * 128 + (((4 * half + ch) ^ (row & 7)) << 4);
                split_store(S + 8 * ch, smem + kScanBsH + o, smem + kScanBsL + o);
            }
        };
        uint64_t* s_mine = is_u ? &sy.s_lo : &sy.s_hi;  // the barrier of this thread's state rows
        store_s();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(s_mine);

        const float* sGc = reinterpret_cast<const float*>(smem + kScanGc);  // [2][64]
        bool alive = true;

        // Output of chunk c (output warps, accumulator rows 64..127), in two
        // parts around the state update that follows it: first the reads of
        // P4's Q S rows, P6 and the gate (after which those buffers may be
        // reused), o = e^{G_t} (Q S)_t + ((M o QK^T) U)_t, its sum of squares
        // and the gated values; then the RMSNorm (sums of squares exchanged
        // with the peer CTA) and the stores.  Every output warp makes the same
        // calls (the named barriers inside must match); after a failure no
        // wait is made.
        float og[32];  // o * norm_w * act(z) of the pending output
        float oss = 0.f;  // sum of o^2 over this thread's 32 value lanes
        float gt_pend = 0.f;  // G_t of this thread's token row in the chunk whose output is pending
        auto output_read = [&](int c, bool alive_in) -> bool {
            const int t = row - 64;
            bool ok = __all_sync(0xffffffffu, alive_in && wait_or_dead(&sy.p6[c & 1], (c >> 1) & 1, sy, 7) &&
                                                  wait_or_dead(&sy.gate, c & 1, sy, 9));
            if (!ok) return false;
            tc_fence_after_sync();
            float a[32];
            const uint32_t d4 = tmem + kTmD4 + (uint32_t)(c & 1) * kP4Cols + lane_off + cl;
            const uint32_t d6 = tmem + kTmD6 + (uint32_t)(c & 1) * 64 + lane_off + cl;
            if constexpr (kSplitP4) {
                tmem_ld32x2(d4, d6, a, og);
            } else {
                float b[32];
                tmem_ld32x3(d4, d4 + 64, d6, a, b, og);
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] += b[j];
            }
            const float eg = exp_ftz(gt_pend);
            oss = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                og[j] = fmaf(eg, a[j], og[j]);
                oss = fmaf(og[j], og[j], oss);
            }
            const float* gb = reinterpret_cast<const float*>(smem + kScanGate) + t * kC;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 v = *reinterpret_cast<const float4*>(gb + ((((cl >> 2) + c4) ^ (t & 15)) << 2));
                og[4 * c4] *= v.x; og[4 * c4 + 1] *= v.y; og[4 * c4 + 2] *= v.z; og[4 * c4 + 3] *= v.w;
            }
            tc_fence_before_sync();
            // the slots of P4_{c+2} and P6_{c+2}, the gate of chunk c+1 and G buffer c%2 may be reused
            mbar_arrive(&sy.d4free[c & 1]);
            return true;
        };
        auto output_finish = [&](int c, bool ok) -> bool {
            const int t = row - 64, s = c & 1, L = chunk_len(c);
            sSq[half][t] = ok ? oss : 0.f;
            group_sync(1, 128);  // the output warps' halves of each row are in sSq
            const float tot = sSq[0][t] + sSq[1][t];
            if (ok && half == 0) {
                // the peer's slot s is free once it has read chunk c-2 from it
                ok = c < 2 || wait_or_dead(&sy.xf[s], ((c - 2) >> 1) & 1, sy, 10, true, peer_dead);
                if (ok) {
                    if (t == 0) mbar_arrive_expect_tx(&sy.x[s], kC * 4);  // arm: the peer's 64 sums
                    st_async_f32(map_to_rank(smem_u32(&sx[s][t]), peer), tot,
                                 map_to_rank(smem_u32(&sy.x[s]), peer));
                }
            }
            ok = ok && wait_or_dead(&sy.x[s], (c >> 1) & 1, sy, 10, false, peer_dead);
            const float peer_tot = sx[s][t];
            group_sync(1, 128);  // both halves have read sx[s] for this chunk
            if (ok && half == 0) mbar_arrive_remote_relaxed(map_to_rank(smem_u32(&sy.xf[s]), peer), peer_tot);
            if (ok && t < L) {  // gated RMSNorm of token t over all d_v lanes
                const float rr = rsqrtf((tot + peer_tot) * (1.f / kD) + p.rms_eps);
                uint4* op = reinterpret_cast<uint4*>(p.out + (size_t)(tok0(c) + t) * hv_n * kD +
                                                     (size_t)h * kD + v0 + cl);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] = og[8 * i + e] * rr;
                    op[i] = pack_bf16x8(y);
                }
            }
            return ok;
        };

        // The compute warps read no global memory inside the loop: the chunk
        // data come into shared memory by the producer's copies, and global
        // loads in flight would hold up every mbarrier arrive (a release)
        // until they land.  U warps leave the loop on a failure; output warps
        // go through every iteration (with no waits) so that their named
        // barriers stay matched.
        for (int c = 0; c < n_ch; ++c) {
            if (!alive && is_u) break;
            // U~ and G of chunk c (the output warps read G of chunk c here, before
            // their arrive for chunk c-1 lets the producer reuse this buffer)
            alive = __all_sync(0xffffffffu, alive && wait_or_dead(&sy.ug, c & 1, sy, 12));
            const float* gc = sGc + (c & 1) * kC;
            // state decay over chunk c (of this thread's key row, per-channel decay)
            const float gam = !alive ? 0.f
                              : kKda ? exp_ftz(reinterpret_cast<const float*>(smem + kScanGl)[(c & 1) * kD + row])
                                     : exp_ftz(gc[chunk_len(c) - 1]);
            float gt_next = 0.f;
            if (!kKda && !is_u && alive) gt_next = gc[row - 64];
            bool out_ok = false;
            if (is_u) {
                // U_c = U~ - W S_c (rows 0..63 of P4_c), U'_c = e^{G_last-G_t} U_c
                const float eu = kKda ? 1.f : exp_ftz(gc[chunk_len(c) - 1] - gc[row]);
                float ut[32];
                const float4* us4 = reinterpret_cast<const float4*>(smem + kScanUt) + ((cl >> 2) * kC + row);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v = us4[i * kC];
                    ut[4 * i] = v.x; ut[4 * i + 1] = v.y; ut[4 * i + 2] = v.z; ut[4 * i + 3] = v.w;
                }
                // warp-uniform: the tensor-memory loads below are warp-collective
                if (!(alive = __all_sync(0xffffffffu, alive && wait_or_dead(&sy.p4, c & 1, sy, 5)))) break;
                tc_fence_after_sync();
                {
                    float a[32];
                    const uint32_t d4 = tmem + kTmD4 + (uint32_t)(c & 1) * kP4Cols + lane_off + cl;
                    if constexpr (kSplitP4) {
                        tmem_ld32(d4, a);
                    } else {
                        float b[32];
                        tmem_ld32x2(d4, d4 + 64, a, b);
#pragma unroll
                        for (int j = 0; j < 32; ++j) a[j] += b[j];
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) ut[j] -= a[j];
                }
                // U' for P7_c (P7_{c-1} has read the last one), then U for P6_c
                // (P6_{c-1} has read U_{c-1}): both readers are done once P4_c
                // is, which the issuer committed after them.  Only U' is on the
                // chain.  The arrive on u also releases the U~ buffer.
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t o = row * 128 + (((4 * half + ch) ^ (row & 7)) << 4);
                    float us[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) us[e] = ut[8 * ch + e] * eu;
                    split_store(us, smem + kScanUp + o, smem + kScanUp + 8192 + o);
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&sy.u);
                // U_c replaces U_{c-1} once P6_{c-1} has read it
                if (c > 0 && !(alive = __all_sync(0xffffffffu, wait_or_dead(&sy.p6[(c - 1) & 1],
                                                                            ((c - 1) >> 1) & 1, sy, 7))))
                    break;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t ob = row * 128 + (((4 * half + ch) ^ (row & 7)) << 4);
                    split_store(ut + 8 * ch, smem + kScanBu + ob, smem + kScanBu + 8192 + ob);
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&sy.u2);
            } else if (c > 0) {
                // the output of chunk c-1, read before this chunk's state update
                out_ok = output_read(c - 1, alive);
            }
            gt_pend = gt_next;
            // S_{c+1} = e^{G_last} S_c + K''^T U_c ; refresh the split copy
            alive = __all_sync(0xffffffffu, alive && wait_or_dead(&sy.p7, c & 1, sy, 6));
            if (alive) {
                tc_fence_after_sync();
                float a[32];
                const uint32_t ds = tmem + kTmDs + lane_off + cl;
                tmem_ld32(ds, a);
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] = fmaf(gam, S[j], a[j]);
                if (c + 1 < n_ch) {
                    store_s();
                    fence_proxy_async_smem();
                    tc_fence_before_sync();
                    mbar_arrive(s_mine);
                }
            }
            if (!is_u && c > 0) alive = output_finish(c - 1, out_ok && alive) && alive;
        }
        if (n_ch > 0 && !is_u) {
            const bool ok = output_read(n_ch - 1, alive);
            alive = output_finish(n_ch - 1, ok && alive) && alive;
        }
        if (alive && p.state_out) {
            float4* dst = reinterpret_cast<float4*>(p.state_out + slab + (size_t)row * kD + v0 + cl);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
        }
        if (!alive) atomicExch(&sy.dead, 1);
    }

    // Unwind: no copy or MMA of this CTA may still be in flight when it leaves.
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (tid == 0) {
        if (sy.n_a4 > 0) mbar_wait(&sy.a4, (sy.n_a4 - 1) & 1);
        if (sy.n_k > 0) mbar_wait(&sy.k, (sy.n_k - 1) & 1);
        if (sy.n_qk > 0) mbar_wait(&sy.qk, (sy.n_qk - 1) & 1);
        if (sy.n_ug > 0) mbar_wait(&sy.ug, (sy.n_ug - 1) & 1);
        if (sy.n_zf > 0) mbar_wait(&sy.zf, (sy.n_zf - 1) & 1);
        if (sy.n_p6 > 0) mbar_wait(&sy.p6[(sy.n_p6 - 1) & 1], ((sy.n_p6 - 1) >> 1) & 1);
        if (sy.n_commits > 0) {
            const uint32_t idx = sy.last_commit >> 1, par = sy.last_commit & 1;
            uint64_t* bar = idx == 0 ? &sy.p4 : &sy.p7;
            mbar_wait(bar, par);
        }
    }
    // No CTA may leave while its peer can still reach its shared memory.
    tc_fence_before_sync();
    __syncthreads();
    cluster_arrive();
    cluster_wait();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kScanThreads, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                  const __grid_constant__ CUtensorMap map_wh, const __grid_constant__ CUtensorMap map_wl,
                  const __grid_constant__ CUtensorMap map_kqh, const __grid_constant__ CUtensorMap map_kql,
                  const __grid_constant__ CUtensorMap map_kwh, const __grid_constant__ CUtensorMap map_kwl,
                  const __grid_constant__ CUtensorMap map_z, ChunkArgs p) {
    // sequences with the most chunks start first: the last wave is shorter
    chunk_scan_body<true, false>(map_qh, map_ql, map_wh, map_wl, map_kqh, map_kql, map_kwh, map_kwl, map_z, p,
                    blockIdx.x / kSplit, p.seq_order ? p.seq_order[blockIdx.y] : (int)blockIdx.y);
}

// The scan of the per-channel decay form (after chunk_prep_kda_kernel).
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kScanThreads, 1)
chunk_scan_kda_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                      const __grid_constant__ CUtensorMap map_wh, const __grid_constant__ CUtensorMap map_wl,
                      const __grid_constant__ CUtensorMap map_kqh, const __grid_constant__ CUtensorMap map_kql,
                      const __grid_constant__ CUtensorMap map_kwh, const __grid_constant__ CUtensorMap map_kwl,
                      const __grid_constant__ CUtensorMap map_z, ChunkArgs p) {
    chunk_scan_body<true, true>(map_qh, map_ql, map_wh, map_wl, map_kqh, map_kql, map_kwh, map_kwl, map_z, p,
                                blockIdx.x / kSplit, p.seq_order ? p.seq_order[blockIdx.y] : (int)blockIdx.y);
}

// ------------------------------------------------------------- chunk_fused
// Both phases in one launch, for batches whose scan alone would leave most of
// the GPU idle (its clusters run one chunk after another).  CTAs [0, n_prep)
// run chunk_prep over every item, chunk-major, and set each item's flag once
// its rows have landed; the other CTAs run chunk_scan, one cluster per
// (sequence, value head), and read a chunk's rows only after its flag is set,
// so the scan of chunk c overlaps the prep of the chunks after it.  Prep CTAs
// never wait for scan CTAs: the launch completes whichever of its CTAs are
// resident at a time.  A prep CTA's control warpgroup hands its registers to
// the eight prep warps (232 each) and leaves.
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kScanThreads, 1)
chunk_fused_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_ql,
                   const __grid_constant__ CUtensorMap map_wh, const __grid_constant__ CUtensorMap map_wl,
                   const __grid_constant__ CUtensorMap map_kqh, const __grid_constant__ CUtensorMap map_kql,
                   const __grid_constant__ CUtensorMap map_kwh, const __grid_constant__ CUtensorMap map_kwl,
                   const __grid_constant__ CUtensorMap map_z, ChunkArgs p, int n_prep) {
    if ((int)blockIdx.x < n_prep) {
        // the control warpgroup leaves: 256 x 232 + 128 x 40 = 384 x 168
        if (threadIdx.x >= kComputeThreads) {
            regs_dec<40>();
            return;
        }
        regs_inc<232>();
        chunk_prep_body(map_qh, map_ql, map_wh, map_wl, map_kqh, map_kql, map_kwh, map_kwl, p,
                        blockIdx.x, n_prep);
    } else {
        const int s = ((int)blockIdx.x - n_prep) / kSplit;  // n_prep is even: clusters stay aligned
        chunk_scan_body<false, false>(map_qh, map_ql, map_wh, map_wl, map_kqh, map_kql, map_kwh, map_kwl, map_z, p,
                        s % p.n_v_heads, s / p.n_v_heads);
    }
}

// ------------------------------------------------------------------- host
size_t chunked_workspace_bytes(int n_seq, const int32_t* cu_host, int n_k_heads, int n_v_heads,
                               int per_channel, ChunkLayout* lay) {
    ChunkLayout l{};
    const size_t pc = per_channel ? 1 : 0;
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
    l.g = off; off = up(off + (pc ? 0 : (size_t)T * n_v_heads * 4));  // per channel: formed by its prep
    l.beta = off; off = up(off + (size_t)T * n_v_heads * 4);
    l.cu_chunks = off; off = up(off + (size_t)(n_seq + 1) * 4);
    l.chunk_info = off; off = up(off + (size_t)chunks * 8);
    l.seq_order = off; off = up(off + (size_t)n_seq * 4);
    // per-channel decay: W rows, then as many rows of Q o e^G
    l.w_hi = off; off = up(off + (1 + pc) * crow * kD * 2);
    l.w_lo = off; off = up(off + (1 + pc) * crow * kD * 2);
    l.u = off; off = up(off + crow * kD * 4);
    l.qk_hi = off; off = up(off + crow * kC * 2);
    l.qk_lo = off; off = up(off + crow * kC * 2);
    // key rows per key head (per value head, decayed, with per-channel decay)
    const size_t krows = pc ? crow : (size_t)chunks * n_k_heads * kC;
    l.kw_hi = off; off = up(off + krows * kD * 2);
    l.kw_lo = off; off = up(off + krows * kD * 2);
    l.gcum = off; off = up(off + (pc ? crow * 2 : crow) * 4);
    l.ready = off; off = up(off + ((size_t)chunks * n_k_heads + 1) * 4);  // + one never set (test hook)
    l.total = off;
    l.n_chunks = static_cast<int>(chunks);
    l.per_channel = per_channel ? 1 : 0;
    if (lay) *lay = l;
    return off;
}

// CTAs of chunk_fused_kernel that can be resident at once (2 x its active
// clusters), per device; 0 when the query fails.  (The per-device caches here
// are atomics: host threads may make their first call on a device at once.)
static int fused_capacity(size_t smem) {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev].load()) {
        cudaFuncSetAttribute(chunk_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2 * kSplit);
        cfg.blockDim = dim3(kScanThreads);
        cfg.dynamicSmemBytes = smem;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, chunk_fused_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            nc = 0;
        }
        cached[dev].store(nc > 0 ? 2 * nc : -1);
    }
    const int cap = cached[dev].load();
    return cap > 0 ? cap : 0;
}

// SMs of the current device (the persistent prep kernel runs one CTA per SM).
static int sm_count() {
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

// A scan launch as the programmatic dependent of the prep kernel before it
// (which triggers at its start): its CTAs may start setting up on SMs the prep
// has left; the copy lane waits for the prep grid before reading its rows.
template <typename Kernel, typename... Args>
static cudaError_t launch_after_prep(Kernel kernel, dim3 grid, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kScanThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
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
    cv.decay_form = a.decay_form;
    cv.per_channel = a.per_channel;
    cv.conv_w = a.conv_w; cv.A_log = a.A_log; cv.dt_bias = a.dt_bias;
    cv.conv_state_in = a.conv_state_in;
    cv.conv_state_out = a.conv_state_out;
    cv.qkv_out = ws + l.qkv_hi;
    cv.qkv_lo_out = ws + l.qkv_lo;
    cv.g_out = reinterpret_cast<float*>(ws + l.g);
    cv.beta_out = reinterpret_cast<float*>(ws + l.beta);
    cv.zero_tail = kC;  // the padding chunk after the last token: read by partial-chunk tiles
    int32_t* cu_chunks = reinterpret_cast<int32_t*>(ws + l.cu_chunks);
    if (a.n_seq > 0) {  // the chunk table, built by one CTA of the prologue
        cv.cu_chunks = cu_chunks;
        cv.chunk_info = reinterpret_cast<int2*>(ws + l.chunk_info);
        cv.ready = reinterpret_cast<int*>(ws + l.ready);
        cv.n_ready = l.n_chunks * hk_n + 1;
        // a longest-first launch order for the two-kernel scan (quadratic in
        // the sequence count, so only for batches of up to 1024 sequences)
        if (a.n_seq > 1 && a.n_seq <= 1024) cv.seq_order = reinterpret_cast<int32_t*>(ws + l.seq_order);
    }
    cudaError_t e = timed_launch("conv_prologue", st, [&] { return launch_conv_prologue(cv, true, st); });
    if (e != cudaSuccess) return e;
    if (a.n_seq == 0) return cudaSuccess;


    ChunkArgs p{};
    p.n_seq = a.n_seq; p.n_tokens = T; p.n_chunks = l.n_chunks;
    p.n_k_heads = hk_n; p.n_v_heads = hv_n; p.act = a.act; p.rms_eps = a.rms_eps;
    p.head_map = a.head_map;
    p.cu_seqlens = a.cu_seqlens; p.cu_chunks = cu_chunks;
    p.chunk_info = reinterpret_cast<const int2*>(ws + l.chunk_info);
    p.seq_order = cv.seq_order;
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
    p.gcum_ws = reinterpret_cast<float*>(ws + l.gcum);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.wait_ns = 2000000000ull;

    // Tensor maps; with no chunk at all (only empty sequences) no kernel
    // dereferences them and they stay zero.
    CUtensorMap m_qh, m_ql, m_wh, m_wl, m_kqh, m_kql, m_kwh, m_kwl, m_z;
    std::memset(&m_qh, 0, sizeof(m_qh));
    m_ql = m_wh = m_wl = m_kqh = m_kql = m_kwh = m_kwl = m_z = m_qh;
    const bool pc = a.per_channel != 0;
    const uint64_t crow = (uint64_t)l.n_chunks * hv_n * kC;
    const uint64_t krows = pc ? crow : (uint64_t)l.n_chunks * hk_n * kC;
    if (pc) {
        p.qt_row0 = static_cast<int>(crow);
        p.gate_a = static_cast<const __nv_bfloat16*>(a.a);
        p.A_log = a.A_log;
        p.dt_bias = a.dt_bias;
        p.decay_form = a.decay_form;
        p.kw_hi = reinterpret_cast<__nv_bfloat16*>(ws + l.kw_hi);
        p.kw_lo = reinterpret_cast<__nv_bfloat16*>(ws + l.kw_lo);
    }
    if (l.n_chunks > 0) {
        if (!make_tma_map_bf16_2d(&m_qh, ws + l.qkv_hi, (uint64_t)T + kC, cd, cd, 64, 64) ||
            !make_tma_map_bf16_2d(&m_ql, ws + l.qkv_lo, (uint64_t)T + kC, cd, cd, 64, 64) ||
            !make_tma_map_bf16_2d(&m_wh, ws + l.w_hi, (pc ? 2 : 1) * crow, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_wl, ws + l.w_lo, (pc ? 2 : 1) * crow, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kqh, ws + l.qk_hi, crow, kC, kC, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kql, ws + l.qk_lo, crow, kC, kC, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kwh, ws + l.kw_hi, krows, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_kwl, ws + l.kw_lo, krows, kD, kD, 64, 64) ||
            !make_tma_map_bf16_2d(&m_z, a.z, (uint64_t)T, (uint64_t)hv_n * kD, (uint64_t)hv_n * kD, 64, 64))
            return cudaErrorInvalidValue;
    }

    const size_t prep_smem = 1024 + kPrepVec + (size_t)R * 4 * kC * 4;
    const size_t scan_smem = 1024 + kScanEnd;
    const size_t scan_smem_kda = 1024 + kScanEndKda;
    const size_t prep_smem_max = 1024 + kPrepVec + 8 * 4 * kC * 4;
    // the kernels' shared-memory opt-in is a per-device setting
    static std::atomic<bool> attrs_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attrs_set[dev].load()) {
        cudaError_t ae = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(prep_smem_max));
        if (ae == cudaSuccess)
            ae = cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(scan_smem));
        if (ae == cudaSuccess)
            ae = cudaFuncSetAttribute(chunk_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(std::max(prep_smem_max, scan_smem)));
        if (ae == cudaSuccess)
            ae = cudaFuncSetAttribute(chunk_scan_kda_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(scan_smem_kda));
        if (ae != cudaSuccess) return ae;
        attrs_set[dev].store(true);
    }
    if (pc) {  // per-channel decay: its prep over (chunk, value head) items, then its scan
        if (l.n_chunks > 0) {
            const int n_kda = l.n_chunks * hv_n;
            CUtensorMap m_a;  // the gate input, a [T, Hv*128] (bf16)
            if (!make_tma_map_bf16_2d(&m_a, a.a, (uint64_t)T, (uint64_t)hv_n * kD, (uint64_t)hv_n * kD, 64, 64))
                return cudaErrorInvalidValue;
            e = timed_launch("chunk_prep_kda", st, [&] {
                return launch_kda_prep(m_qh, m_ql, m_kqh, m_kql, m_a, p, std::min(n_kda, sm_count()), st);
            });
            if (e != cudaSuccess) return e;
        }
        return timed_launch("chunk_scan_kda", st, [&] {
            // launched after its prep completes: as a dependent starting in the
            // prep's tail, its 64 CTAs measured slower (641 -> 650 us a step),
            // all placed on the SMs that happened to finish first
            chunk_scan_kda_kernel<<<dim3(hv_n * kSplit, a.n_seq), kScanThreads, scan_smem_kda, st>>>(
                m_qh, m_ql, m_wh, m_wl, m_kqh, m_kql, m_kwh, m_kwl, m_z, p);
            return cudaGetLastError();
        });
    }
    const int n_items = l.n_chunks * hk_n;
    // One fused launch when the scan's clusters leave at least 32 CTA slots
    // of the co-resident capacity for prep (GDN_PREFILL_FUSED=0 turns it off).
    const int scan_ctas = hv_n * kSplit * a.n_seq;
    int n_prep = 0;
    const char* fz = std::getenv("GDN_PREFILL_FUSED");
    if (n_items > 0 && !(fz && fz[0] == '0')) {
        const int cap = fused_capacity(std::max(prep_smem_max, scan_smem));
        if (scan_ctas + 32 <= cap) n_prep = std::min(cap - scan_ctas, (n_items + 1) & ~1);
    }
    if (n_prep > 0) {
        p.ready = reinterpret_cast<int*>(ws + l.ready);
        if (a.stall) {  // the flag after the items' ones: cleared by the prologue, never set
            p.stall_flag = p.ready + n_items;
            p.wait_ns = 1000000ull;
        }
        return timed_launch("chunk_fused", st, [&] {
            chunk_fused_kernel<<<dim3(n_prep + scan_ctas), kScanThreads, std::max(prep_smem, scan_smem),
                                 st>>>(m_qh, m_ql, m_wh, m_wl, m_kqh, m_kql, m_kwh, m_kwl, m_z, p, n_prep);
            return cudaGetLastError();
        });
    }
    if (l.n_chunks > 0) {
        e = timed_launch("chunk_prep", st, [&] {
            chunk_prep_kernel<<<dim3(std::min(n_items, sm_count())), kChunkThreads, prep_smem, st>>>(
                m_qh, m_ql, m_wh, m_wl, m_kqh, m_kql, m_kwh, m_kwl, p);
            return cudaGetLastError();
        });
        if (e != cudaSuccess) return e;
    }
    e = timed_launch("chunk_scan", st, [&] {
        return launch_after_prep(chunk_scan_kernel, dim3(hv_n * kSplit, a.n_seq), scan_smem, st, m_qh, m_ql,
                                 m_wh, m_wl, m_kqh, m_kql, m_kwh, m_kwl, m_z, p);
    });
    return e;
}

cudaError_t read_device_error(int* code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    }
    // the projection GEMM's word (codes 20..23), the recurrent kernel's (30),
    // the per-channel prep's (13, 14)
    int gemm = 0, rec = 0, kda = 0;
    if (e == cudaSuccess) e = read_gemm_error(&gemm, reset);
    if (e == cudaSuccess) e = read_rec_error(&rec, reset);
    if (e == cudaSuccess) e = read_kda_error(&kda, reset);
    if (e == cudaSuccess && *code == 0) *code = gemm ? gemm : rec ? rec : kda;
    return e;
}

}  // namespace gdn
