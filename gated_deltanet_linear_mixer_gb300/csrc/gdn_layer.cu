// One GDN layer's prefill around the core: the input projections, the core
// (gdn_prefill) and the output projection.  qwen.rs gdn_forward runs
// in_proj_qkv, in_proj_z, in_proj_b and in_proj_a as one linear_multi over the
// hidden states, then the core, then out_proj over the gated-norm output.
// Here the four input projections are one launch of this library's tcgen05
// GEMM (each written in the layout the core reads: x [T, CD], z [T, Hv*dv],
// a, b [T, Hv]), and out_proj a second launch over the core's output y.
#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {
// Records the thread's error message (defined with the other entry points).
gdn_status set_error(gdn_status st, const char* fn, const char* fmt, ...);
// GDN_ERR_INJECTED when the environment variable GDN_FAULT lists `site`.
gdn_status inject_fault(const char* site, const char* fn);
}  // namespace gdn

namespace {

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct LayerLayout {
    size_t x, z, a, b, y, core, total;
};

LayerLayout layer_layout(const gdn_dims* d, size_t T, size_t core_bytes) {
    const size_t cd = 2 * (size_t)d->n_k_heads * d->d_k + (size_t)d->n_v_heads * d->d_v;
    const size_t vd = (size_t)d->n_v_heads * d->d_v, hv = (size_t)d->n_v_heads;
    LayerLayout l{};
    size_t off = 0;
    l.x = off; off = up256(off + T * cd * 2);
    l.z = off; off = up256(off + T * vd * 2);
    l.a = off; off = up256(off + T * hv * 2);
    l.b = off; off = up256(off + T * hv * 2);
    l.y = off; off = up256(off + T * vd * 2);
    l.core = off; off = up256(off + core_bytes);
    l.total = off;
    return l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" gdn_status gdn_layer_prefill_workspace_size(const gdn_dims* dims, int32_t hidden,
                                                       int32_t n_seq,
                                                       const int32_t* cu_seqlens_host,
                                                       size_t* bytes) {
    const char* fn = "gdn_layer_prefill_workspace_size";
    if (!bytes) return gdn::set_error(GDN_ERR_INVALID_ARG, fn, "bytes is NULL");
    if (hidden < 8 || hidden % 8 != 0)
        return gdn::set_error(GDN_ERR_INVALID_ARG, fn, "hidden must be a positive multiple of 8 (got %d)",
                              hidden);
    size_t core = 0;
    gdn_status st = gdn_prefill_workspace_size(dims, n_seq, cu_seqlens_host, &core);
    if (st != GDN_OK) return st;
    const size_t T = n_seq > 0 ? (size_t)cu_seqlens_host[n_seq] : 0;
    *bytes = layer_layout(dims, T, core).total;
    return GDN_OK;
}

extern "C" gdn_status gdn_layer_prefill(const gdn_dims* dims, const gdn_params* params,
                                        const gdn_proj* proj, int32_t hidden, int32_t n_seq,
                                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                        const void* h_in, const float* initial_state,
                                        float* final_state, const void* conv_state_in,
                                        void* conv_state_out, void* h_out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    const char* fn = "gdn_layer_prefill";
    size_t need = 0;
    gdn_status st = gdn_layer_prefill_workspace_size(dims, hidden, n_seq, cu_seqlens_host, &need);
    if (st != GDN_OK) return st;
    if (dims->dtype != GDN_DTYPE_BF16)
        return gdn::set_error(GDN_ERR_UNSUPPORTED, fn, "the layer runs on bf16 activations only");
    if (dims->decay_per_channel)
        return gdn::set_error(GDN_ERR_UNSUPPORTED, fn, "per-channel decays are not built into the layer");
    if (!proj || !proj->w_qkv || !proj->w_z || !proj->w_a || !proj->w_b || !proj->w_out)
        return gdn::set_error(GDN_ERR_INVALID_ARG, fn, "a projection weight is NULL");
    if (!aligned16(proj->w_qkv) || !aligned16(proj->w_z) || !aligned16(proj->w_a) ||
        !aligned16(proj->w_b) || !aligned16(proj->w_out))
        return gdn::set_error(GDN_ERR_INVALID_ARG, fn, "projection weights must be 16-byte aligned");
    if (n_seq == 0) return GDN_OK;
    if (!h_in || !h_out || !aligned16(h_in) || !aligned16(h_out))
        return gdn::set_error(GDN_ERR_INVALID_ARG, fn, "h_in and h_out must be 16-byte aligned, non-NULL");
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return gdn::set_error(GDN_ERR_WORKSPACE, fn,
                              "a 256-byte aligned workspace of %zu bytes is needed (%zu given)", need,
                              workspace ? workspace_bytes : (size_t)0);
    if ((st = gdn::inject_fault("layer", fn)) != GDN_OK) return st;
    const int T = cu_seqlens_host[n_seq];
    size_t core_bytes = 0;
    gdn_prefill_workspace_size(dims, n_seq, cu_seqlens_host, &core_bytes);
    const LayerLayout l = layer_layout(dims, (size_t)T, core_bytes);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int cd = 2 * dims->n_k_heads * dims->d_k + dims->n_v_heads * dims->d_v;
    const int vd = dims->n_v_heads * dims->d_v, hv = dims->n_v_heads;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // the input projections, one launch: x = h W_qkv^T, z = h W_z^T, a = h W_a^T, b = h W_b^T
    gdn::GemmLaunch in{};
    in.a = h_in; in.m = T; in.k = hidden; in.n_seg = 4;
    in.seg[0] = {proj->w_qkv, ws + l.x, cd, cd};
    in.seg[1] = {proj->w_z, ws + l.z, vd, vd};
    in.seg[2] = {proj->w_a, ws + l.a, hv, hv};
    in.seg[3] = {proj->w_b, ws + l.b, hv, hv};
    cudaError_t e = gdn::timed_launch("proj_in", s, [&] { return gdn::launch_gemm_bf16(in, s); });
    if (e != cudaSuccess)
        return gdn::set_error(GDN_ERR_CUDA, fn, "input projection launch failed: %s", cudaGetErrorString(e));
    st = gdn_prefill(dims, params, n_seq, cu_seqlens, cu_seqlens_host, ws + l.x, ws + l.z, ws + l.a,
                     ws + l.b, conv_state_in, conv_state_out, initial_state, final_state, ws + l.y,
                     ws + l.core, core_bytes, stream);
    if (st != GDN_OK) return st;
    // out_proj over the core's output y
    gdn::GemmLaunch out{};
    out.a = ws + l.y; out.m = T; out.k = vd; out.n_seg = 1;
    out.seg[0] = {proj->w_out, h_out, hidden, hidden};
    e = gdn::timed_launch("proj_out", s, [&] { return gdn::launch_gemm_bf16(out, s); });
    if (e != cudaSuccess)
        return gdn::set_error(GDN_ERR_CUDA, fn, "output projection launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}
