// The projections around the core on tcgen05 tensor cores: C = A W^T with A
// [M, K] and W [N, K] bf16 row-major (the [out_features, in_features] layout of
// qwen.rs's linear weights), fp32 accumulation in tensor memory, bf16 output.
// One launch computes several products that share A (qwen.rs gdn_forward runs
// in_proj_qkv, in_proj_z, in_proj_b and in_proj_a as one linear_multi over the
// hidden states): output segment s takes its columns from W_s and writes them
// to C_s with its own row stride, so each projection lands in the layout its
// consumer reads (x [T, CD] is the conv prologue's input as it stands).
//
// Persistent CTAs, one per SM, walk the 128 x BN output tiles (BN = 256, or 32
// for the narrow a and b projections), M fastest so that neighbouring CTAs
// share a weight tile in L2.  Warp roles:
//   warp 0     one lane loads A and W tiles (TMA, 128-byte swizzle) into a
//              4-stage ring of 64-wide K blocks
//   warp 1     one lane issues the MMAs (M=128, N=BN, K=16) into one of two
//              accumulators in tensor memory and commits each stage back to
//              the loader and each finished tile to the epilogue
//   warps 2-5  the epilogue: tensor memory -> registers -> bf16 -> global,
//              one accumulator while the MMAs fill the other
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

constexpr int kBM = 128, kBK = 64, kStages = 4, kMaxBN = 256, kMaxSeg = 4;
constexpr uint32_t kStageA = kBM * kBK * 2;       // 16 KB
constexpr uint32_t kStageB = kMaxBN * kBK * 2;    // 32 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr int kGemmThreads = 192;
constexpr size_t kGemmSmem = 1024 + (size_t)kStages * kStageBytes;

__device__ int g_gemm_error = 0;
__device__ __forceinline__ void gemm_fail(int code) { atomicCAS(&g_gemm_error, 0, code); }

struct GemmArgs {
    int m, k, n_seg, tiles_m;
    int seg_tile0[kMaxSeg + 1];  // first global N-tile of each segment; [n_seg] = all N-tiles
    int bn[kMaxSeg], n[kMaxSeg], ldc[kMaxSeg];
    __nv_bfloat16* c[kMaxSeg];
};

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                    const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                    const __grid_constant__ CUtensorMap map_b3, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_slot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 128);
        }
        fence_barrier_init();
        for (const CUtensorMap* m : {&map_a, &map_b0, &map_b1, &map_b2, &map_b3}) tma_prefetch_desc(m);
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const int n_tiles = g.tiles_m * g.seg_tile0[g.n_seg];
    const int nk = (g.k + kBK - 1) / kBK;
    // tile t -> output segment s, M-tile mt, N-tile nt within the segment
    auto tile_info = [&](int t, int& s, int& mt, int& nt) {
        const int ntg = t / g.tiles_m;
        mt = t - ntg * g.tiles_m;
        s = 0;
        while (s + 1 < g.n_seg && g.seg_tile0[s + 1] <= ntg) ++s;
        nt = ntg - g.seg_tile0[s];
    };

    if (warp == 0) {
        if (lane == 0) {  // loader
            uint32_t kbg = 0;
            uint32_t armed[kStages] = {};
            bool ok = true;
            for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
                int s, mt, nt;
                tile_info(t, s, mt, nt);
                const CUtensorMap* mb = s == 0 ? &map_b0 : s == 1 ? &map_b1 : s == 2 ? &map_b2 : &map_b3;
                const int bn = g.bn[s];
                for (int kb = 0; kb < nk; ++kb, ++kbg) {
                    const int st = kbg % kStages;
                    if (kbg >= kStages && !(ok = mbar_wait(&empty[st], ((kbg / kStages) - 1) & 1))) break;
                    mbar_arrive_expect_tx(&full[st], kStageA + (uint32_t)bn * kBK * 2);
                    tma_load_2d(smem + st * kStageBytes, &map_a, &full[st], kb * kBK, mt * kBM);
                    tma_load_2d(smem + st * kStageBytes + kStageA, mb, &full[st], kb * kBK, nt * bn);
                    armed[st] += 1;
                }
            }
            if (!ok) gemm_fail(20);
            for (int st = 0; st < kStages; ++st)  // no copy may be in flight when the CTA leaves
                if (armed[st] && !mbar_wait(&full[st], (armed[st] - 1) & 1)) gemm_fail(21);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            uint32_t kbg = 0;
            bool ok = true;
            uint64_t* last = nullptr;
            uint32_t last_par = 0;
            const uint32_t sa = smem_u32(smem);
            int i = 0;
            for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++i) {
                int s, mt, nt;
                tile_info(t, s, mt, nt);
                const int ab = i & 1;
                if (i >= 2 && !(ok = mbar_wait(&acc_empty[ab], ((i >> 1) - 1) & 1))) break;
                tc_fence_after_sync();
                const uint32_t idesc = idesc_bf16_f32(kBM, g.bn[s]);
                const uint32_t d = tmem + (uint32_t)ab * 256;
                for (int kb = 0; kb < nk; ++kb, ++kbg) {
                    const int st = kbg % kStages;
                    if (!(ok = mbar_wait(&full[st], (kbg / kStages) & 1))) break;
                    tc_fence_after_sync();
                    const uint64_t da = desc_kmajor_sw128(sa + st * kStageBytes);
                    const uint64_t db = desc_kmajor_sw128(sa + st * kStageBytes + kStageA);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_bf16(d, da + 2 * k, db + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&empty[st]);  // the stage is free once these MMAs are done
                    last = &empty[st];
                    last_par = (kbg / kStages) & 1;
                }
                if (!ok) break;
                mma_commit(&acc_full[ab]);
                last = &acc_full[ab];
                last_par = (i >> 1) & 1;
            }
            if (!ok) gemm_fail(22);
            if (last && !mbar_wait(last, last_par)) gemm_fail(22);
        }
    } else {  // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31
        const int q = warp & 3;
        int i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            int s, mt, nt;
            tile_info(t, s, mt, nt);
            const int ab = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (i >> 1) & 1))) {
                if (lane == 0) gemm_fail(23);
                break;
            }
            tc_fence_after_sync();
            const int row = mt * kBM + 32 * q + lane;
            const int bn = g.bn[s], nvalid = min(bn, g.n[s] - nt * bn);
            __nv_bfloat16* crow = g.c[s] + (size_t)row * g.ldc[s] + (size_t)nt * bn;
            const bool vec = (g.ldc[s] & 7) == 0;
            for (int j = 0; j < bn / 32; ++j) {
                float v[32];
                tmem_ld32(tmem + (uint32_t)ab * 256 + 32 * j + ((32u * q) << 16), v);
                if (row >= g.m) continue;
                const int c0 = 32 * j;
                if (vec && c0 + 32 <= nvalid) {
                    uint4* dst = reinterpret_cast<uint4*>(crow + c0);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u] = make_uint4(pack_bf16_pair(v[8 * u], v[8 * u + 1]),
                                            pack_bf16_pair(v[8 * u + 2], v[8 * u + 3]),
                                            pack_bf16_pair(v[8 * u + 4], v[8 * u + 5]),
                                            pack_bf16_pair(v[8 * u + 6], v[8 * u + 7]));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c0 + e < nvalid) crow[c0 + e] = __float2bfloat16_rn(v[e]);
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&acc_empty[ab]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

int sm_count_gemm() {
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

}  // namespace

cudaError_t launch_gemm_bf16(const GemmLaunch& l, cudaStream_t st) {
    if (l.n_seg < 1 || l.n_seg > kMaxSeg || l.m < 0 || l.k < 1) return cudaErrorInvalidValue;
    if (l.m == 0) return cudaSuccess;
    GemmArgs g{};
    g.m = l.m;
    g.k = l.k;
    g.n_seg = l.n_seg;
    g.tiles_m = (l.m + kBM - 1) / kBM;
    CUtensorMap ma, mb[kMaxSeg];
    std::memset(&ma, 0, sizeof(ma));
    for (auto& m : mb) m = ma;
    if (!make_tma_map_bf16_2d(&ma, l.a, (uint64_t)l.m, (uint64_t)l.k, (uint64_t)l.k, kBM, kBK))
        return cudaErrorInvalidValue;
    int tiles_n = 0;
    for (int s = 0; s < l.n_seg; ++s) {
        const GemmSegment& sg = l.seg[s];
        const int bn = sg.n >= 128 ? 256 : 32;
        if (sg.n < 1 || !make_tma_map_bf16_2d(&mb[s], sg.w, (uint64_t)sg.n, (uint64_t)l.k, (uint64_t)l.k,
                                              bn, kBK))
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
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
        cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kGemmSmem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true);
    }
    const int n_tiles = g.tiles_m * tiles_n;
    const int grid = std::min(n_tiles, sm_count_gemm());
    gemm_bf16_tn_kernel<<<grid, kGemmThreads, kGemmSmem, st>>>(ma, mb[0], mb[1], mb[2], mb[3], g);
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
