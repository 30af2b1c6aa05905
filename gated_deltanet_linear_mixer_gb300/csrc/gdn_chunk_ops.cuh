// Device helpers shared by the chunked prefill kernels (scalar and per-channel
// decay): bf16 (hi, lo) split arithmetic for tensor-core operands, the prep
// role's barriers, the warp-level products of the triangular solve and the
// solve itself, and the publication of a finished prep item.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {

using namespace tc;

constexpr int kC = kChunkTokens;   // chunk length
constexpr int kD = 128;            // d_k = d_v on this path

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
// Barriers of the prep role: named barrier 1 over its eight warps (256
// threads), so that a launch may carry more warps than prep uses.
__device__ __forceinline__ void prep_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// Every prep thread learns whether any of them passed v != 0.
__device__ __forceinline__ bool prep_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}
// Uniform decision after a bounded wait: every prep thread learns whether any
// thread's wait gave up.
__device__ __forceinline__ bool prep_failed(bool ok) { return prep_any(!ok); }

// Split arithmetic.  Every tensor-core operand is carried as a pair of bf16
// tiles, hi = bf16(x) and lo = bf16(x - hi), which together hold ~16
// significant bits; a product A.B is formed as hi.hi + hi.lo + lo.hi with
// fp32 accumulation (the dropped lo.lo term is ~2^-16 relative).  The gated
// outputs are heavy-tailed (up to ~50x their RMS), so plain bf16 operands
// (2^-9 relative) would put the largest outputs' error far above 2e-2 of the
// output RMS.
__device__ __forceinline__ void split_store(const float* f, uint8_t* hi, uint8_t* lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // hi rounded once per pair; lo = the exact remainder, rounded
        h[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
        l[i] = pack_bf16x2(f[2 * i] - __uint_as_float(h[i] << 16),
                           f[2 * i + 1] - __uint_as_float(h[i] & 0xFFFF0000u));
    }
    *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
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

// The solve's fp32 64 x 64 tiles (A, T) are row-major with their 16-byte
// chunks XOR-swizzled by the row: chunk c of row r sits at chunk c ^ (r & 15).
// Row vectors and the column reads of mma fragments are both free of bank
// conflicts.  Offset (in floats) of column col within row r:
__device__ __forceinline__ int swz_col(int r, int col) {
    return (((col >> 2) ^ (r & 15)) << 2) + (col & 3);
}

// Warp-level bf16 tensor-core product (m16n8k16, fp32 accumulation) for the
// 16 x 16 blocks of the triangular solve.  Operands are split like the
// tcgen05 ones (hi = bf16(x), lo = bf16(x - hi)) and every product is
// hi.hi + hi.lo + lo.hi.  Fragment layouts (lane = 4 g + q):
//   A 16 x 16: a0 (g, 2q..2q+1), a1 (g+8, 2q..), a2 (g, 2q+8..), a3 (g+8, 2q+8..)
//   B 16 x 8:  b0 (k = 2q..2q+1, n = g), b1 (k = 2q+8..2q+9, n = g)
//   C 16 x 8:  c0, c1 (g, 2q..2q+1), c2, c3 (g+8, 2q..2q+1)
// so the two C tiles of a 16 x 16 result are, element for element, the A
// fragment of a following product.
struct SplitA { uint32_t h[4], l[4]; };
struct SplitB { uint32_t h[2], l[2]; };

__device__ __forceinline__ void split2(float x, float y, uint32_t& h, uint32_t& l) {
    h = pack_bf16x2(x, y);
    l = pack_bf16x2(x - __uint_as_float(h << 16), y - __uint_as_float(h & 0xFFFF0000u));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// A fragment of block (bi, bj) of a swizzled tile given by its row pointers.
template <class Rows>
__device__ __forceinline__ SplitA solve_load_a(Rows rows, int bi, int bj, int lane) {
    const int g = lane >> 2, q = lane & 3;
    SplitA a;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = 16 * bi + g + 8 * (k & 1), c = 16 * bj + 2 * q + 8 * (k >> 1);
        const float2 v = *reinterpret_cast<const float2*>(rows(r) + swz_col(r, c));
        split2(v.x, v.y, a.h[k], a.l[k]);
    }
    return a;
}
// D (16 x 16, two C tiles) = A B (+ D), B = block (bk, bn) of a swizzled tile.
template <class Rows>
__device__ __forceinline__ void solve_mma(float (*d)[4], const SplitA& a, Rows rows, int bk, int bn,
                                          int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * bn + 8 * nt + g;
        SplitB b;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = 16 * bk + 2 * q + 8 * k;
            split2(rows(r)[swz_col(r, c)], rows(r + 1)[swz_col(r + 1, c)], b.h[k], b.l[k]);
        }
        mma16816(d[nt], a.h, b.h[0], b.h[1]);
        mma16816(d[nt], a.h, b.l[0], b.l[1]);
        mma16816(d[nt], a.l, b.h[0], b.h[1]);
    }
}
__device__ __forceinline__ SplitA solve_c_to_a(const float (*d)[4]) {
    SplitA a;
    split2(d[0][0], d[0][1], a.h[0], a.l[0]);
    split2(d[0][2], d[0][3], a.h[1], a.l[1]);
    split2(d[1][0], d[1][1], a.h[2], a.l[2]);
    split2(d[1][2], d[1][3], a.h[3], a.l[3]);
    return a;
}


// An item is published (p.ready non-null) once all of its workspace writes
// have landed: the TMA stores completed, then a gpu-scope release that also
// covers the other threads' stores (they precede it through the CTA barrier).
__device__ __forceinline__ void publish_item(int* flag) {
    bulk_wait_all();
    fence_proxy_async_global();
    __threadfence();
    st_release_gpu(flag, 1);
}

// T = (I + A)^-1 of one head's strictly lower triangular 64 x 64 A (fp32, rows
// given by rowsA / rowsT, 16-byte chunks swizzled as swz_col), by 16 x 16
// blocks on four warps (w = 0..3) that share named barrier `bar` (128
// threads).  Diagonal blocks T_ii = (I + A_ii)^-1 by forward substitution in
// fp32, one warp each; then with Y_ij = T_ii A_ij (i > j),
//   T_ij = -sum_{k=j}^{i-1} Y_ik T_kj,
// one block distance i - j per step, on the warp tensor cores.  Blocks above
// the diagonal are not written.
template <class RowsA, class RowsT>
__device__ __forceinline__ void solve_unit_lower(RowsA rowsA, RowsT rowsT, uint32_t bar, int w, int lane) {
    {   // T_ww, column j per lane (lanes 16..31 repeat lanes 0..15)
        const int i = w, j = lane & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            // row r of A_ii as 16-byte chunks (those left of the diagonal)
            const int row = 16 * i + r;
            float a16[16];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                if (4 * c4 < r) {
                    const float4 v4 = *reinterpret_cast<const float4*>(
                        rowsA(row) + (((4 * i + c4) ^ (row & 15)) << 2));
                    a16[4 * c4] = v4.x; a16[4 * c4 + 1] = v4.y;
                    a16[4 * c4 + 2] = v4.z; a16[4 * c4 + 3] = v4.w;
                }
            }
            float acc = r == j ? 1.f : 0.f;
#pragma unroll
            for (int s2 = 0; s2 < r; ++s2) acc = fmaf(-a16[s2], x[s2], acc);
            x[r] = acc;
            asm volatile("" ::: "memory");  // one row's loads at a time
        }
        if (lane < 16) {
#pragma unroll
            for (int r = 0; r < 16; ++r) rowsT(16 * i + r)[swz_col(16 * i + r, 16 * i + j)] = x[r];
        }
    }
    group_sync(bar, 128);
    SplitA y[3];  // Y_wk, k < w
    if (w > 0) {
        const SplitA tw = solve_load_a(rowsT, w, w, lane);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            if (k < w) {
                float d[2][4] = {};
                solve_mma(d, tw, rowsA, w, k, lane);
                y[k] = solve_c_to_a(d);
            }
        }
    }
#pragma unroll
    for (int dist = 1; dist < 4; ++dist) {
        if (dist > 1) group_sync(bar, 128);  // T blocks of distance < dist are stored
        if (w >= dist) {
            const int j = w - dist;
            float d[2][4] = {};
#pragma unroll
            for (int k = 0; k < 3; ++k)
                if (k >= j && k < w) solve_mma(d, y[k], rowsT, k, j, lane);
            const int g = lane >> 2, q = lane & 3;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int r0 = 16 * w + g, c = 16 * j + 8 * nt + 2 * q;
                *reinterpret_cast<float2*>(rowsT(r0) + swz_col(r0, c)) =
                    make_float2(-d[nt][0], -d[nt][1]);
                *reinterpret_cast<float2*>(rowsT(r0 + 8) + swz_col(r0 + 8, c)) =
                    make_float2(-d[nt][2], -d[nt][3]);
            }
        }
    }
}

}  // namespace gdn
