// The projections around the core on tcgen05 tensor cores: C = A W^T with A
// [M, K] and W [N, K] bf16 row-major (the [out_features, in_features] layout of
// qwen.rs's linear weights), fp32 accumulation in tensor memory, bf16 output.
// One launch computes several products that share A (qwen.rs gdn_forward runs
// in_proj_qkv, in_proj_z, in_proj_b and in_proj_a as one linear_multi over the
// hidden states): output segment s takes its columns from W_s and writes them
// to C_s with its own row stride, so each projection lands in the layout its
// consumer reads (x [T, CD] is the conv prologue's input as it stands).
//
// Clusters of two CTAs on neighbouring SMs compute 256 x BN output tiles with
// the pair form of the tensor-core MMA (cta_group::2): each CTA stages its
// own 128 rows of A and its own half of the BN weight rows, and one MMA of
// the even CTA multiplies the pair's whole 256 x BN x 16 block, each CTA's
// tensor memory receiving its 128 output rows.  Per SM that halves the
// weight tile a K step moves through L2 and shared memory against a one-CTA
// 128 x BN tile.  Persistent pairs walk the tiles (BN = 256, or 64 for the
// narrow a and b projections), M fastest so that neighbouring pairs share a
// weight tile in L2.  Warp roles, in both CTAs unless stated:
//   warp 0     one lane loads this CTA's A and W tiles (TMA, 128-byte
//              swizzle) into a 6-stage ring of 64-wide K blocks; every copy
//              completes on the even CTA's stage barrier
//   warp 1     (even CTA) one lane issues the pair MMAs into one of two
//              accumulators and commits each stage back to both loaders and
//              each finished tile to both epilogues
//   warps 2-5  the epilogue: tensor memory -> registers -> bf16 -> a
//              swizzled 32 x 64 staging tile per warp (two, alternating) ->
//              TMA store, one accumulator while the MMAs fill the other; the
//              odd CTA's threads release the accumulator on the even CTA's
//              barrier as soon as they have read it.  (Stores straight from
//              registers, one row per thread, cost a fifth of the launch.)
//              An output whose row stride or base the TMA cannot take is
//              written with plain stores instead.
// Every wait is bounded (2 s); a wait that gives up records a code (20..23) in
// this file's device error word and its role stops.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
#include "gdn_tma_host.h"

namespace gdn {

using namespace tc;

namespace {

#ifndef GDN_GEMM_STAGES
#define GDN_GEMM_STAGES 6
#endif
constexpr int kBM = 128, kBK = 64, kStages = GDN_GEMM_STAGES, kMaxBN = 256, kMaxSeg = 4;
constexpr uint32_t kStageA = kBM * kBK * 2;           // 16 KB: this CTA's 128 rows of A
constexpr uint32_t kStageB = (kMaxBN / 2) * kBK * 2;  // 16 KB: this CTA's half of the W rows
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr uint32_t kStgBytes = 32 * 64 * 2;           // one epilogue staging tile: 32 rows x 128 B
constexpr int kGemmThreads = 192;
constexpr size_t kGemmSmem = 1024 + (size_t)kStages * kStageBytes + 4 * 2 * kStgBytes;

__device__ int g_gemm_error = 0;
__device__ __forceinline__ void gemm_fail(int code) { atomicCAS(&g_gemm_error, 0, code); }

struct GemmArgs {
    int m, k, n_seg, tiles_m;    // tiles_m: 256-row tiles
    int seg_tile0[kMaxSeg + 1];  // first global N-tile of each segment; [n_seg] = all N-tiles
    int bn[kMaxSeg], n[kMaxSeg], ldc[kMaxSeg];
    int c_tma[kMaxSeg];          // 1: segment s is written through map_c[s]
    __nv_bfloat16* c[kMaxSeg];
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                    const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                    const __grid_constant__ CUtensorMap map_b3, const __grid_constant__ CUtensorMap map_c0,
                    const __grid_constant__ CUtensorMap map_c1, const __grid_constant__ CUtensorMap map_c2,
                    const __grid_constant__ CUtensorMap map_c3, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    // full: used in the even CTA only (both CTAs' copies complete on it);
    // empty, acc_full: in both, signalled by the even CTA's commits;
    // acc_empty: in the even CTA, released by both epilogues.
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_slot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 2 * 128);
        }
        fence_barrier_init();
        for (const CUtensorMap* m : {&map_a, &map_b0, &map_b1, &map_b2, &map_b3}) tma_prefetch_desc(m);
        for (int s = 0; s < g.n_seg; ++s)
            if (g.c_tma[s]) tma_prefetch_desc(s == 0 ? &map_c0 : s == 1 ? &map_c1 : s == 2 ? &map_c2 : &map_c3);
    }
    if (warp == 1) tmem_alloc_pair(&tmem_slot, 512);
    tc_fence_before_sync();
    cluster_arrive();  // the peer's barriers are initialised before anyone signals them
    cluster_wait();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int n_tiles = g.tiles_m * g.seg_tile0[g.n_seg];
    const int nk = (g.k + kBK - 1) / kBK;
    // tile t -> output segment s, 256-row M-tile mt, N-tile nt within the segment
    auto tile_info = [&](int t, int& s, int& mt, int& nt) {
        const int ntg = t / g.tiles_m;
        mt = t - ntg * g.tiles_m;
        s = 0;
        while (s + 1 < g.n_seg && g.seg_tile0[s + 1] <= ntg) ++s;
        nt = ntg - g.seg_tile0[s];
    };

    if (warp == 0) {
        if (lane == 0) {  // loader
            uint32_t full_even[kStages];
            for (int st = 0; st < kStages; ++st) full_even[st] = map_to_rank(smem_u32(&full[st]), 0);
            uint32_t kbg = 0;
            uint32_t armed[kStages] = {};
            bool ok = true;
            for (int t = pair; ok && t < n_tiles; t += n_pairs) {
                int s, mt, nt;
                tile_info(t, s, mt, nt);
                const CUtensorMap* mb = s == 0 ? &map_b0 : s == 1 ? &map_b1 : s == 2 ? &map_b2 : &map_b3;
                const int half = g.bn[s] >> 1;
                for (int kb = 0; kb < nk; ++kb, ++kbg) {
                    const int st = kbg % kStages;
                    if (kbg >= kStages && !(ok = mbar_wait(&empty[st], ((kbg / kStages) - 1) & 1))) break;
                    // the even CTA arms its barrier with both CTAs' bytes; a copy
                    // of the odd CTA may land first (the count dips below zero)
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&full[st], 2 * (kStageA + (uint32_t)half * kBK * 2));
                        armed[st] += 1;
                    }
                    uint8_t* sa = smem + st * kStageBytes;
                    tma_load_2d_pair(sa, &map_a, full_even[st], kb * kBK, mt * 2 * kBM + (int)rank * kBM);
                    tma_load_2d_pair(sa + kStageA, mb, full_even[st], kb * kBK, nt * g.bn[s] + (int)rank * half);
                }
            }
            if (!ok) gemm_fail(20);
            // no copy of this pair may be in flight when the even CTA leaves
            for (int st = 0; st < kStages; ++st)
                if (armed[st] && !mbar_wait(&full[st], (armed[st] - 1) & 1)) gemm_fail(21);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {  // MMA issuer
            uint32_t kbg = 0;
            bool ok = true;
            uint64_t* last = nullptr;
            uint32_t last_par = 0;
            const uint32_t sa = smem_u32(smem);
            int i = 0;
            for (int t = pair; ok && t < n_tiles; t += n_pairs, ++i) {
                int s, mt, nt;
                tile_info(t, s, mt, nt);
                const int ab = i & 1;
                if (i >= 2 && !(ok = mbar_wait_cluster(&acc_empty[ab], ((i >> 1) - 1) & 1))) break;
                tc_fence_after_sync();
                const uint32_t idesc = idesc_bf16_f32(2 * kBM, g.bn[s]);
                const uint32_t d = tmem + (uint32_t)ab * 256;
                for (int kb = 0; kb < nk; ++kb, ++kbg) {
                    const int st = kbg % kStages;
                    if (!(ok = mbar_wait(&full[st], (kbg / kStages) & 1))) break;
                    tc_fence_after_sync();
                    const uint64_t da = desc_kmajor_sw128(sa + st * kStageBytes);
                    const uint64_t db = desc_kmajor_sw128(sa + st * kStageBytes + kStageA);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_bf16_pair(d, da + 2 * k, db + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit_pair(&empty[st], 0x3);  // both CTAs' stage is free once these are done
                    last = &empty[st];
                    last_par = (kbg / kStages) & 1;
                }
                if (!ok) break;
                mma_commit_pair(&acc_full[ab], 0x3);
                last = &acc_full[ab];
                last_par = (i >> 1) & 1;
            }
            if (!ok) gemm_fail(22);
            if (last && !mbar_wait(last, last_par)) gemm_fail(22);
        }
    } else {  // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31
        const int q = warp & 3;
        const uint32_t acc_empty_even[2] = {map_to_rank(smem_u32(&acc_empty[0]), 0),
                                            map_to_rank(smem_u32(&acc_empty[1]), 0)};
        uint8_t* stg = smem + kStages * kStageBytes + q * 2 * kStgBytes;  // this warp's two tiles
        uint32_t n_stores = 0;
        int i = 0;
        for (int t = pair; t < n_tiles; t += n_pairs, ++i) {
            int s, mt, nt;
            tile_info(t, s, mt, nt);
            const int ab = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (i >> 1) & 1))) {
                if (lane == 0) gemm_fail(23);
                break;
            }
            tc_fence_after_sync();
            const int row0 = mt * 2 * kBM + (int)rank * kBM + 32 * q;  // this warp's first row
            const int bn = g.bn[s], nvalid = min(bn, g.n[s] - nt * bn);
            const uint32_t tacc = tmem + (uint32_t)ab * 256 + ((32u * q) << 16);
            if (g.c_tma[s]) {
                const CUtensorMap* mc = s == 0 ? &map_c0 : s == 1 ? &map_c1 : s == 2 ? &map_c2 : &map_c3;
                for (int j = 0; j < bn / 64; ++j) {
                    float v[64];
                    tmem_ld64(tacc + 64 * j, v);
                    if (j == bn / 64 - 1) {  // the accumulator is read: release it
                        tc_fence_before_sync();
                        if (rank == 0) mbar_arrive(&acc_empty[ab]);
                        else mbar_arrive_remote(acc_empty_even[ab]);
                    }
                    if (row0 >= g.m || 64 * j >= nvalid) continue;  // wholly outside C (warp-uniform)
                    uint8_t* buf = stg + (n_stores & 1) * kStgBytes;
                    if (n_stores >= 2) {  // the store that last read this tile is done with it
                        if (lane == 0) bulk_wait_read_1();
                        __syncwarp();
                    }
                    // row `lane`, 16-byte chunk u at chunk u ^ (lane % 8): the 128-byte swizzle
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<uint4*>(buf + lane * 128 + ((u ^ (lane & 7)) << 4)) =
                            make_uint4(pack_bf16_pair(v[8 * u], v[8 * u + 1]), pack_bf16_pair(v[8 * u + 2], v[8 * u + 3]),
                                       pack_bf16_pair(v[8 * u + 4], v[8 * u + 5]), pack_bf16_pair(v[8 * u + 6], v[8 * u + 7]));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {  // rows >= m and columns >= n are clipped by the map
                        tma_store_2d(mc, buf, nt * bn + 64 * j, row0);
                        bulk_commit();
                    }
                    ++n_stores;
                }
            } else {
                const int row = row0 + lane;
                __nv_bfloat16* crow = g.c[s] + (size_t)row * g.ldc[s] + (size_t)nt * bn;
                for (int j = 0; j < bn / 32; ++j) {
                    float v[32];
                    tmem_ld32(tacc + 32 * j, v);
                    if (row >= g.m || 32 * j >= nvalid) continue;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (32 * j + e < nvalid) crow[32 * j + e] = __float2bfloat16_rn(v[e]);
                }
                tc_fence_before_sync();
                if (rank == 0) mbar_arrive(&acc_empty[ab]);
                else mbar_arrive_remote(acc_empty_even[ab]);
            }
        }
        if (lane == 0) bulk_wait_all();  // no store may still read the staging tiles
        __syncwarp();
    }
    // both CTAs' MMAs, copies and remote arrivals are done before either leaves
    tc_fence_before_sync();
    cluster_arrive();
    cluster_wait();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// Clusters of gemm_bf16_tn_kernel that can be resident at once, per device
// (the persistent grid launches no more pairs than this); 0 if the query fails.
int gemm_pair_capacity() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev].load()) {
        int nc = 0;
        if (cudaFuncSetAttribute(gemm_bf16_tn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmem)) == cudaSuccess) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(kGemmThreads);
            cfg.dynamicSmemBytes = kGemmSmem;
            if (cudaOccupancyMaxActiveClusters(&nc, gemm_bf16_tn_kernel, &cfg) != cudaSuccess) nc = 0;
        }
        cudaGetLastError();
        cached[dev].store(nc > 0 ? nc : -1);
    }
    const int cap = cached[dev].load();
    return cap > 0 ? cap : 0;
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmLaunch& l, cudaStream_t st) {
    if (l.n_seg < 1 || l.n_seg > kMaxSeg || l.m < 0 || l.k < 1) return cudaErrorInvalidValue;
    if (l.m == 0) return cudaSuccess;
    GemmArgs g{};
    g.m = l.m;
    g.k = l.k;
    g.n_seg = l.n_seg;
    g.tiles_m = (l.m + 2 * kBM - 1) / (2 * kBM);
    CUtensorMap ma, mb[kMaxSeg];
    std::memset(&ma, 0, sizeof(ma));
    for (auto& m : mb) m = ma;
    if (!make_tma_map_bf16_2d(&ma, l.a, (uint64_t)l.m, (uint64_t)l.k, (uint64_t)l.k, kBM, kBK))
        return cudaErrorInvalidValue;
    int tiles_n = 0;
    for (int s = 0; s < l.n_seg; ++s) {
        const GemmSegment& sg = l.seg[s];
        const int bn = sg.n >= 128 ? 256 : 64;  // each CTA of a pair loads bn / 2 weight rows
        if (sg.n < 1 || !make_tma_map_bf16_2d(&mb[s], sg.w, (uint64_t)sg.n, (uint64_t)l.k, (uint64_t)l.k,
                                              bn / 2, kBK))
            return cudaErrorInvalidValue;
        g.seg_tile0[s] = tiles_n;
        g.bn[s] = bn;
        g.n[s] = sg.n;
        g.ldc[s] = sg.ldc;
        g.c[s] = static_cast<__nv_bfloat16*>(sg.c);
        tiles_n += (sg.n + bn - 1) / bn;
    }
    g.seg_tile0[l.n_seg] = tiles_n;
    for (int s = l.n_seg; s < kMaxSeg; ++s) mb[s] = mb[0];  // unused
    // output maps: 32 x 64 boxes; a segment whose base or row pitch the TMA
    // cannot take (16-byte alignment) is written with plain stores
    CUtensorMap mc[kMaxSeg];
    for (int s = 0; s < kMaxSeg; ++s) mc[s] = ma;
    for (int s = 0; s < l.n_seg; ++s) {
        const GemmSegment& sg = l.seg[s];
        g.c_tma[s] = (reinterpret_cast<uintptr_t>(sg.c) % 16 == 0) && (sg.ldc % 8 == 0) && sg.ldc >= sg.n &&
                     make_tma_map_bf16_2d(&mc[s], sg.c, (uint64_t)l.m, (uint64_t)sg.n, (uint64_t)sg.ldc, 32, 64);
    }
    const int pairs_max = gemm_pair_capacity();
    if (pairs_max < 1) return cudaErrorLaunchOutOfResources;
    const int n_tiles = g.tiles_m * tiles_n;
    const int pairs = std::min(n_tiles, pairs_max);
    gemm_bf16_tn_kernel<<<2 * pairs, kGemmThreads, kGemmSmem, st>>>(ma, mb[0], mb[1], mb[2], mb[3], mc[0], mc[1], mc[2],
                                                                  mc[3], g);
    return cudaGetLastError();
}

cudaError_t read_gemm_error(int* code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemm_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
    }
    return e;
}

}  // namespace gdn
