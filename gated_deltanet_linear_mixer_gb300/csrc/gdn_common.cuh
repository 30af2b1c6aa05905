// Device helpers shared by the GDN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// ---------------------------------------------------------------- scalar I/O
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// A 16-byte vector of activations: 4 floats or 8 bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static uint4 load_raw(const float* p) {
        return *reinterpret_cast<const uint4*>(p);
    }
    __device__ __forceinline__ static void unpack(uint4 v, float* out) {
        out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
        out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static void load(const float* p, float* out) {
        float4 v = *reinterpret_cast<const float4*>(p);
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
    __device__ __forceinline__ static void store(float* p, const float* in) {
        *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static uint4 load_raw(const __nv_bfloat16* p) {
        return *reinterpret_cast<const uint4*>(p);
    }
    __device__ __forceinline__ static void unpack(uint4 v, float* out) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* out) {
        uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* in) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ------------------------------------------------------------- the method's
// scalar functions (qwen.rs DeltaRule::run / gdn_forward; cpu.rs deltanet)
// The hardware's approximate exponential, base-2 logarithm and reciprocal, in
// their flush-to-zero forms: the non-flushing forms (what __expf, __logf and
// __fdividef compile to) measured slower in the exponential-heavy kernels.
// Results that would be subnormal (below 1.2e-38) become 0.
__device__ __forceinline__ float exp_ftz(float x) {  // e^x = 2^(x log2 e)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}
__device__ __forceinline__ float log_ftz(float x) {  // ln x = log2 x ln 2
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y * 0.6931471805599453f;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// sigmoid and SiLU with those: relative error ~1e-6 over the range the gates
// see, far below both tolerances, at a fraction of the precise functions'
// cost.  For x below about -88 e^-x overflows and the reciprocal is 0 (the
// exact values are below 1e-38 there).
__device__ __forceinline__ float sigmoidf_(float x) { return rcp_ftz(1.0f + exp_ftz(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x * rcp_ftz(1.0f + exp_ftz(-x)); }
// softplus: identity above 20, else ln(1 + e^x)
__device__ __forceinline__ float softplusf_(float x) { return x > 20.0f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float gatef_(float z, int act) {
    return act == 1 ? sigmoidf_(z) : siluf_(z);
}
// log-decay g = -exp(A_log) * softplus(a + dt_bias)
// Log-decay g of one token and value head; A is log A (form 0) or the decay
// coefficient itself (form 1, the GGUF ssm_a).
__device__ __forceinline__ float log_decay(float a, float A, float dt_bias, int form) {
    return (form ? A : -expf(A)) * softplusf_(a + dt_bias);
}

// Key head of value head h (tiled: h % Hk; contiguous: h / R), and the r-th
// value head of key head hk (R = Hv / Hk value heads per key head).
__device__ __forceinline__ int key_head(int h, int R, int Hk, int tiled) { return tiled ? h % Hk : h / R; }
__device__ __forceinline__ int value_head(int hk, int r, int R, int Hk, int tiled) {
    return tiled ? hk + Hk * r : hk * R + r;
}

// Two floats rounded to bf16 (nearest even) and packed, first in the low half.
__device__ __forceinline__ uint32_t pack_bf16_pair(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ------------------------------------------------------------ reductions
template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// The sequence that packed token t belongs to: largest i with cu[i] <= t
// (empty sequences are skipped).  cu has n+1 entries, cu[0] = 0.
__device__ __forceinline__ int seq_of_token(const int32_t* __restrict__ cu, int n, int t) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace gdn
