// C-ABI entry points of libgdn (declared in include/gdn.h): host-side
// validation of every argument, error reporting, and kernel dispatch on the
// caller's stream.  No entry point allocates device memory.
#include <cmath>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

thread_local char g_err[512] = "";

gdn_status fail(gdn_status st, const char* fn, const char* fmt, ...) {
    int n = std::snprintf(g_err, sizeof(g_err), "%s: ", fn);
    if (n < 0) n = 0;
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err + n, sizeof(g_err) - (size_t)n, fmt, ap);
    va_end(ap);
    return st;
}

gdn_status cuda_status(cudaError_t e, const char* fn, const char* what) {
    if (e == cudaSuccess) return GDN_OK;
    return fail(GDN_ERR_CUDA, fn, "%s failed: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the comma-separated list in the environment variable GDN_FAULT names
// `site` (or "all").  Read on every call, so a test can set and clear it.
bool fault_listed(const char* site) {
    const char* v = std::getenv("GDN_FAULT");
    if (!v || !*v) return false;
    const size_t n = std::strlen(site);
    for (const char* p = v; *p;) {
        const char* e = p;
        while (*e && *e != ',') ++e;
        const size_t len = static_cast<size_t>(e - p);
        if ((len == n && std::strncmp(p, site, n) == 0) || (len == 3 && std::strncmp(p, "all", 3) == 0))
            return true;
        p = *e ? e + 1 : e;
    }
    return false;
}

// Host-side fault injection: a call whose site GDN_FAULT lists fails with
// GDN_ERR_INJECTED after validating its arguments and before it enqueues any
// work, so that a caller's failure path can be exercised without a GPU fault.
gdn_status injected(const char* site, const char* fn) {
    if (!fault_listed(site)) return GDN_OK;
    return fail(GDN_ERR_INJECTED, fn, "fault injected at site '%s' (GDN_FAULT); nothing was enqueued",
                site);
}

bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

gdn_status check_dims(const gdn_dims* d, const char* fn) {
    if (!d) return fail(GDN_ERR_INVALID_ARG, fn, "dims is NULL");
    if (d->n_k_heads < 1 || d->n_v_heads < 1)
        return fail(GDN_ERR_INVALID_ARG, fn, "head counts must be >= 1 (Hk=%d, Hv=%d)",
                    d->n_k_heads, d->n_v_heads);
    if (d->n_v_heads % d->n_k_heads != 0)
        return fail(GDN_ERR_UNSUPPORTED, fn, "n_v_heads (%d) must be a multiple of n_k_heads (%d)",
                    d->n_v_heads, d->n_k_heads);
    if (!head_dim_ok(d->d_k) || !head_dim_ok(d->d_v))
        return fail(GDN_ERR_UNSUPPORTED, fn, "d_k and d_v must be 32, 64 or 128 (got %d, %d)",
                    d->d_k, d->d_v);
    if (d->conv_k < 2 || d->conv_k > 4)
        return fail(GDN_ERR_UNSUPPORTED, fn, "conv_k must be 2..4 (got %d)", d->conv_k);
    if (d->dtype != GDN_DTYPE_F32 && d->dtype != GDN_DTYPE_BF16)
        return fail(GDN_ERR_INVALID_ARG, fn, "dtype %d is not a gdn_dtype", d->dtype);
    if (d->act != GDN_ACT_SILU && d->act != GDN_ACT_SIGMOID)
        return fail(GDN_ERR_INVALID_ARG, fn, "act %d is not a gdn_act", d->act);
    if (d->head_map != GDN_HEADS_CONTIGUOUS && d->head_map != GDN_HEADS_TILED)
        return fail(GDN_ERR_INVALID_ARG, fn, "head_map %d is not a gdn_head_map", d->head_map);
    if (d->decay_form != GDN_DECAY_A_LOG && d->decay_form != GDN_DECAY_COEF)
        return fail(GDN_ERR_INVALID_ARG, fn, "decay_form %d is not a gdn_decay_form", d->decay_form);
    if (d->decay_per_channel != 0 && d->decay_per_channel != 1)
        return fail(GDN_ERR_INVALID_ARG, fn, "decay_per_channel must be 0 or 1");
    if (!(d->l2_eps > 0.f) || !std::isfinite(d->l2_eps) || !(d->rms_eps > 0.f) ||
        !std::isfinite(d->rms_eps))
        return fail(GDN_ERR_INVALID_ARG, fn, "eps values must be finite and > 0");
    const long long cd = 2LL * d->n_k_heads * d->d_k + (long long)d->n_v_heads * d->d_v;
    if (cd > (1 << 20)) return fail(GDN_ERR_UNSUPPORTED, fn, "conv_dim %lld is too large", cd);
    return GDN_OK;
}

long long conv_dim(const gdn_dims* d) {
    return 2LL * d->n_k_heads * d->d_k + (long long)d->n_v_heads * d->d_v;
}

bool ranges_overlap(const void* a, const void* b, size_t bytes) {
    if (!a || !b) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
}

// The bf16 prefill (scalar or per-channel decay) takes the chunked
// tensor-core path unless every sequence has at most kShortPrefill tokens (a replayed verify prefix, a batch of
// decode-sized prompts): then the token-recurrent kernel, which streams each
// state once and has no chunk to fill, is the faster one.
constexpr int kShortPrefill = 16;
bool use_chunked(const gdn_dims* d, int n_seq, const int32_t* cu_host) {
    if (!gdn::chunked_supported(d->d_k, d->d_v, d->n_k_heads, d->n_v_heads, d->dtype == GDN_DTYPE_BF16))
        return false;
    for (int i = 0; i < n_seq; ++i)
        if (cu_host[i + 1] - cu_host[i] > kShortPrefill) return true;
    return false;
}

gdn_status check_params(const gdn_params* p, bool need_norm, const char* fn) {
    if (!p) return fail(GDN_ERR_INVALID_ARG, fn, "params is NULL");
    if (!p->conv_w || !p->A_log || !p->dt_bias || (need_norm && !p->norm_w))
        return fail(GDN_ERR_INVALID_ARG, fn, "a parameter pointer is NULL");
    return GDN_OK;
}

// Validates the host copy of cu_seqlens; returns the total token count.
gdn_status check_cu(int32_t n_seq, const int32_t* cu_dev, const int32_t* cu_host, int* total,
                    const char* fn) {
    if (n_seq < 0) return fail(GDN_ERR_INVALID_ARG, fn, "n_seq must be >= 0 (got %d)", n_seq);
    if (n_seq > GDN_MAX_SEQUENCES)
        return fail(GDN_ERR_UNSUPPORTED, fn, "n_seq %d is above GDN_MAX_SEQUENCES (%d)", n_seq,
                    GDN_MAX_SEQUENCES);
    *total = 0;
    if (n_seq == 0) return GDN_OK;
    if (!cu_dev || !cu_host) return fail(GDN_ERR_INVALID_ARG, fn, "cu_seqlens pointer is NULL");
    if (cu_host[0] != 0) return fail(GDN_ERR_INVALID_ARG, fn, "cu_seqlens[0] must be 0");
    for (int i = 0; i < n_seq; ++i)
        if (cu_host[i + 1] < cu_host[i])
            return fail(GDN_ERR_INVALID_ARG, fn, "cu_seqlens decreases at index %d", i + 1);
    *total = cu_host[n_seq];
    return GDN_OK;
}


// ------------------------------------------------------------------ timing
// Optional per-kernel device timing: when enabled, every kernel launch the
// library makes is bracketed by two CUDA events recorded on the launching
// stream.  gdn_timing_report() waits for the events and sums per kernel.
struct TimedLaunch {
    const char* name;
    cudaEvent_t start, stop;
};
struct KernelTotal {
    std::string name;
    long long launches = 0;
    double total_ms = 0.0;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimedLaunch> g_pending;
std::vector<cudaEvent_t> g_event_pool;
std::vector<KernelTotal> g_totals;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void drain_pending_locked() {
    for (auto& r : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) == cudaSuccess &&
            cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
            KernelTotal* t = nullptr;
            for (auto& k : g_totals)
                if (k.name == r.name) t = &k;
            if (!t) {
                g_totals.push_back(KernelTotal{r.name});
                t = &g_totals.back();
            }
            t->launches += 1;
            t->total_ms += ms;
        }
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_pending.clear();
}


}  // namespace

namespace gdn {

gdn_status inject_fault(const char* site, const char* fn) { return injected(site, fn); }

gdn_status set_error(gdn_status st, const char* fn, const char* fmt, ...) {
    int n = std::snprintf(g_err, sizeof(g_err), "%s: ", fn);
    if (n < 0) n = 0;
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err + n, sizeof(g_err) - (size_t)n, fmt, ap);
    va_end(ap);
    return st;
}

void* timing_start(const char* name, cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (!g_timing_on) return nullptr;
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) {
        if (a) g_event_pool.push_back(a);
        if (b) g_event_pool.push_back(b);
        return nullptr;
    }
    cudaEventRecord(a, stream);
    g_pending.push_back({name, a, b});
    return reinterpret_cast<void*>(g_pending.size());  // 1-based index
}

void timing_stop(void* handle, cudaStream_t stream) {
    if (!handle) return;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    const size_t idx = reinterpret_cast<size_t>(handle) - 1;
    if (idx < g_pending.size()) cudaEventRecord(g_pending[idx].stop, stream);
}

}  // namespace gdn

using gdn::timed_launch;

extern "C" {

gdn_status gdn_timing_enable(int32_t enable) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    drain_pending_locked();
    if (enable) g_totals.clear();
    g_timing_on = enable != 0;
    return GDN_OK;
}

size_t gdn_timing_report(char* buf, size_t buf_len) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    drain_pending_locked();
    std::string text;
    char line[256];
    for (auto& k : g_totals) {
        std::snprintf(line, sizeof(line), "%s %lld %.6f\n", k.name.c_str(), k.launches, k.total_ms);
        text += line;
    }
    if (buf && buf_len > 0) {
        const size_t n = text.size() < buf_len - 1 ? text.size() : buf_len - 1;
        std::memcpy(buf, text.data(), n);
        buf[n] = '\0';
    }
    return text.size() + 1;
}

gdn_status gdn_device_error(int32_t* code, int32_t reset) {
    const char* fn = "gdn_device_error";
    if (!code) return fail(GDN_ERR_INVALID_ARG, fn, "code is NULL");
    int v = 0;
    gdn_status st = cuda_status(gdn::read_device_error(&v, reset != 0), fn, "reading the error word");
    *code = v;
    return st;
}

gdn_status gdn_sync_status(void* stream) {
    const char* fn = "gdn_sync_status";
    gdn_status st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), fn,
                                "synchronizing the stream");
    if (st != GDN_OK) return st;
    int code = 0;
    if ((st = cuda_status(gdn::read_device_error(&code, true), fn, "reading the error word")) != GDN_OK)
        return st;
    if (code)
        return fail(GDN_ERR_TIMEOUT, fn,
                    "a bounded device wait gave up (wait code %d%s); the "
                    "outputs and states written by the calls since the last check are invalid",
                    code, code == 11 ? ": a scan waited for a chunk's prep rows" : "");
    g_err[0] = '\0';
    return GDN_OK;
}

const char* gdn_last_error(void) { return g_err; }

const char* gdn_version(void) { return "gdn-gb300 0.1 (sm_103a)"; }

gdn_status gdn_conv(const gdn_dims* dims, const gdn_params* params, int32_t n_seq,
                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, const void* x,
                    const void* a, const void* b, const void* conv_state_in,
                    void* conv_state_out, void* qkv_out, float* g_out, float* beta_out,
                    void* stream) {
    const char* fn = "gdn_conv";
    gdn_status st;
    if ((st = check_dims(dims, fn)) != GDN_OK) return st;
    if ((st = check_params(params, false, fn)) != GDN_OK) return st;
    int total = 0;
    if ((st = check_cu(n_seq, cu_seqlens, cu_seqlens_host, &total, fn)) != GDN_OK) return st;
    g_err[0] = '\0';
    if (total == 0 && !conv_state_out) return GDN_OK;
    if (total > 0 && (!x || !a || !b || !qkv_out || !g_out || !beta_out))
        return fail(GDN_ERR_INVALID_ARG, fn, "an input or output pointer is NULL");
    if ((x && !aligned16(x)) || (qkv_out && !aligned16(qkv_out)))
        return fail(GDN_ERR_INVALID_ARG, fn, "x and qkv_out must be 16-byte aligned");
    if ((st = injected("conv", fn)) != GDN_OK) return st;
    const bool bf16 = dims->dtype == GDN_DTYPE_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    gdn::ConvArgs p{};
    p.n_seq = n_seq; p.n_tokens = total;
    p.n_k_heads = dims->n_k_heads; p.n_v_heads = dims->n_v_heads;
    p.d_k = dims->d_k; p.d_v = dims->d_v; p.conv_k = dims->conv_k; p.l2_eps = dims->l2_eps;
    p.cu_seqlens = cu_seqlens; p.x = x; p.a = a; p.b = b; p.decay_form = dims->decay_form;
    p.per_channel = dims->decay_per_channel;
    p.conv_w = params->conv_w; p.A_log = params->A_log; p.dt_bias = params->dt_bias;
    p.conv_state_in = conv_state_in; p.qkv_out = qkv_out; p.g_out = g_out; p.beta_out = beta_out;
    if ((st = cuda_status(timed_launch("conv_prologue", s, [&] { return gdn::launch_conv_prologue(p, bf16, s); }), fn, "conv prologue launch")) != GDN_OK)
        return st;
    if (conv_state_out && n_seq > 0) {
        gdn::ConvStateArgs c{};
        c.n_seq = n_seq; c.n_k_heads = dims->n_k_heads; c.n_v_heads = dims->n_v_heads;
        c.d_k = dims->d_k; c.d_v = dims->d_v; c.conv_k = dims->conv_k;
        c.cu_seqlens = cu_seqlens; c.x = x; c.conv_state_in = conv_state_in;
        c.conv_state_out = conv_state_out;
        if ((st = cuda_status(timed_launch("conv_state", s, [&] { return gdn::launch_conv_state(c, bf16, s); }), fn, "conv state launch")) != GDN_OK)
            return st;
    }
    return GDN_OK;
}

gdn_status gdn_prefill_workspace_size(const gdn_dims* dims, int32_t n_seq,
                                      const int32_t* cu_seqlens_host, size_t* bytes) {
    const char* fn = "gdn_prefill_workspace_size";
    gdn_status st;
    if ((st = check_dims(dims, fn)) != GDN_OK) return st;
    if (!bytes) return fail(GDN_ERR_INVALID_ARG, fn, "bytes is NULL");
    if (n_seq < 0) return fail(GDN_ERR_INVALID_ARG, fn, "n_seq must be >= 0");
    if (n_seq > 0 && !cu_seqlens_host) return fail(GDN_ERR_INVALID_ARG, fn, "cu_seqlens_host is NULL");
    *bytes = 0;
    if (n_seq > 0) {
        int total = 0;
        if ((st = check_cu(n_seq, cu_seqlens_host, cu_seqlens_host, &total, fn)) != GDN_OK)
            return st;
        if (!use_chunked(dims, n_seq, cu_seqlens_host)) return GDN_OK;
        *bytes = gdn::chunked_workspace_bytes(n_seq, cu_seqlens_host, dims->n_k_heads,
                                              dims->n_v_heads, dims->decay_per_channel, nullptr);
    }
    g_err[0] = '\0';
    return GDN_OK;
}

gdn_status gdn_prefill(const gdn_dims* dims, const gdn_params* params, int32_t n_seq,
                       const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                       const void* x, const void* z, const void* a, const void* b,
                       const void* conv_state_in, void* conv_state_out,
                       const float* initial_state, float* final_state, void* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "gdn_prefill";
    gdn_status st;
    if ((st = check_dims(dims, fn)) != GDN_OK) return st;
    if ((st = check_params(params, true, fn)) != GDN_OK) return st;
    int total = 0;
    if ((st = check_cu(n_seq, cu_seqlens, cu_seqlens_host, &total, fn)) != GDN_OK) return st;
    if (total > 0 && (!x || !z || !a || !b || !out))
        return fail(GDN_ERR_INVALID_ARG, fn, "an input or output pointer is NULL");
    if ((x && !aligned16(x)) || (z && !aligned16(z)) || (out && !aligned16(out)) ||
        (initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
        return fail(GDN_ERR_INVALID_ARG, fn, "x, z, out and the states must be 16-byte aligned");
    if (dims->decay_per_channel && a && !aligned16(a))
        return fail(GDN_ERR_INVALID_ARG, fn, "with per-channel decay, a must be 16-byte aligned");
    size_t need = 0;
    if ((st = gdn_prefill_workspace_size(dims, n_seq, cu_seqlens_host, &need)) != GDN_OK) return st;
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(GDN_ERR_WORKSPACE, fn, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    g_err[0] = '\0';
    if ((st = injected("prefill", fn)) != GDN_OK) return st;
    if (n_seq == 0) return GDN_OK;
    const bool bf16 = dims->dtype == GDN_DTYPE_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    bool conv_done = false;
    if (use_chunked(dims, n_seq, cu_seqlens_host)) {
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(GDN_ERR_WORKSPACE, fn, "workspace must be 256-byte aligned");
        gdn::ChunkLaunch c{};
        c.n_seq = n_seq; c.n_tokens = total; c.n_k_heads = dims->n_k_heads;
        c.n_v_heads = dims->n_v_heads; c.conv_k = dims->conv_k; c.act = dims->act;
        c.head_map = dims->head_map; c.decay_form = dims->decay_form;
        c.per_channel = dims->decay_per_channel;
        c.l2_eps = dims->l2_eps; c.rms_eps = dims->rms_eps; c.cu_seqlens = cu_seqlens;
        c.x = x; c.z = z; c.a = a; c.b = b;
        c.conv_w = params->conv_w; c.A_log = params->A_log; c.dt_bias = params->dt_bias;
        c.norm_w = params->norm_w; c.conv_state_in = conv_state_in;
        c.state_in = initial_state; c.state_out = final_state; c.out = out;
        c.workspace = workspace;
        c.stall = fault_listed("stall_scan") ? 1 : 0;
        // the new conv history comes from the prologue's launch unless it is
        // updated in place (the prologue still reads the old one)
        if (conv_state_out && !ranges_overlap(conv_state_in, conv_state_out,
                                              (size_t)n_seq * conv_dim(dims) * (dims->conv_k - 1) * 2)) {
            c.conv_state_out = conv_state_out;
            conv_done = true;
        }
        gdn::chunked_workspace_bytes(n_seq, cu_seqlens_host, dims->n_k_heads, dims->n_v_heads,
                                     dims->decay_per_channel, &c.layout);
        if ((st = cuda_status(gdn::launch_chunked_prefill(c, s), fn, "chunked prefill launch")) !=
            GDN_OK)
            return st;
    } else {
    gdn::RecurrentArgs r{};
    r.n_seq = n_seq; r.n_k_heads = dims->n_k_heads; r.n_v_heads = dims->n_v_heads;
    r.conv_k = dims->conv_k; r.act = dims->act; r.l2_eps = dims->l2_eps; r.rms_eps = dims->rms_eps;
    r.head_map = dims->head_map; r.decay_form = dims->decay_form;
    r.per_channel = dims->decay_per_channel;
    r.cu_seqlens = cu_seqlens; r.uniform_T = 0;
    r.x = x; r.z = z; r.a = a; r.b = b;
    r.conv_w = params->conv_w; r.A_log = params->A_log; r.dt_bias = params->dt_bias;
    r.norm_w = params->norm_w; r.conv_state_in = conv_state_in;
    r.state_in = initial_state; r.state_out = final_state; r.inter = nullptr; r.out = out;
    if ((st = cuda_status(timed_launch("recurrent", s, [&] { return gdn::launch_recurrent(r, dims->d_k, dims->d_v, bf16, s); }), fn,
                          "recurrent launch")) != GDN_OK)
        return st;
    }
    if (conv_state_out && !conv_done) {
        gdn::ConvStateArgs c{};
        c.n_seq = n_seq; c.n_k_heads = dims->n_k_heads; c.n_v_heads = dims->n_v_heads;
        c.d_k = dims->d_k; c.d_v = dims->d_v; c.conv_k = dims->conv_k;
        c.cu_seqlens = cu_seqlens; c.x = x; c.conv_state_in = conv_state_in;
        c.conv_state_out = conv_state_out;
        c.pdl = 1;  // after the recurrent kernel: starts in its tail
        if ((st = cuda_status(timed_launch("conv_state", s, [&] { return gdn::launch_conv_state(c, bf16, s); }), fn, "conv state launch")) != GDN_OK)
            return st;
    }
    return GDN_OK;
}

gdn_status gdn_decode(const gdn_dims* dims, const gdn_params* params, int32_t n_seq, int32_t T,
                      const void* x, const void* z, const void* a, const void* b, float* state,
                      void* conv_state, float* inter_states, void* out, void* stream) {
    const char* fn = "gdn_decode";
    gdn_status st;
    if ((st = check_dims(dims, fn)) != GDN_OK) return st;
    if ((st = check_params(params, true, fn)) != GDN_OK) return st;
    if (n_seq < 0 || n_seq > GDN_MAX_SEQUENCES)
        return fail(GDN_ERR_INVALID_ARG, fn, "n_seq must be 0..GDN_MAX_SEQUENCES (%d) (got %d)",
                    GDN_MAX_SEQUENCES, n_seq);
    if (T < 1 || T > 16) return fail(GDN_ERR_INVALID_ARG, fn, "T must be 1..16 (got %d)", T);
    g_err[0] = '\0';
    if (n_seq == 0) return GDN_OK;
    if (!x || !z || !a || !b || !state || !out)
        return fail(GDN_ERR_INVALID_ARG, fn, "an input or output pointer is NULL");
    if (!aligned16(x) || !aligned16(z) || !aligned16(out) || !aligned16(state) ||
        (inter_states && !aligned16(inter_states)))
        return fail(GDN_ERR_INVALID_ARG, fn, "x, z, out and the states must be 16-byte aligned");
    if ((st = injected("decode", fn)) != GDN_OK) return st;
    const bool bf16 = dims->dtype == GDN_DTYPE_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    gdn::RecurrentArgs r{};
    r.n_seq = n_seq; r.n_k_heads = dims->n_k_heads; r.n_v_heads = dims->n_v_heads;
    r.conv_k = dims->conv_k; r.act = dims->act; r.l2_eps = dims->l2_eps; r.rms_eps = dims->rms_eps;
    r.head_map = dims->head_map; r.decay_form = dims->decay_form;
    r.per_channel = dims->decay_per_channel;
    r.cu_seqlens = nullptr; r.uniform_T = T;
    r.x = x; r.z = z; r.a = a; r.b = b;
    r.conv_w = params->conv_w; r.A_log = params->A_log; r.dt_bias = params->dt_bias;
    r.norm_w = params->norm_w; r.conv_state_in = conv_state;
    r.state_in = state;
    r.state_out = inter_states ? nullptr : state;
    r.inter = inter_states;
    r.out = out;
    if ((st = cuda_status(timed_launch("recurrent", s, [&] {
             return gdn::launch_recurrent(r, dims->d_k, dims->d_v, bf16, s);
         }), fn, "recurrent launch")) != GDN_OK)
        return st;
    if (conv_state && !inter_states) {
        gdn::ConvStateArgs c{};
        c.n_seq = n_seq; c.n_k_heads = dims->n_k_heads; c.n_v_heads = dims->n_v_heads;
        c.d_k = dims->d_k; c.d_v = dims->d_v; c.conv_k = dims->conv_k;
        c.cu_seqlens = nullptr; c.uniform_T = T; c.x = x;
        c.conv_state_in = conv_state; c.conv_state_out = conv_state;
        c.pdl = 1;  // starts in the recurrent kernel's tail
        if ((st = cuda_status(timed_launch("conv_state", s, [&] { return gdn::launch_conv_state(c, bf16, s); }), fn, "conv state launch")) != GDN_OK)
            return st;
    }
    return GDN_OK;
}

gdn_status gdn_verify(const gdn_dims* dims, const gdn_params* params, int32_t n_seq, int32_t T,
                      const void* x, const void* z, const void* a, const void* b,
                      const float* state, const void* conv_state, void* out, void* stream) {
    const char* fn = "gdn_verify";
    gdn_status st;
    if ((st = check_dims(dims, fn)) != GDN_OK) return st;
    if ((st = check_params(params, true, fn)) != GDN_OK) return st;
    if (n_seq < 0 || n_seq > GDN_MAX_SEQUENCES)
        return fail(GDN_ERR_INVALID_ARG, fn, "n_seq must be 0..GDN_MAX_SEQUENCES (%d) (got %d)",
                    GDN_MAX_SEQUENCES, n_seq);
    if (T < 1 || T > 16) return fail(GDN_ERR_INVALID_ARG, fn, "T must be 1..16 (got %d)", T);
    g_err[0] = '\0';
    if (n_seq == 0) return GDN_OK;
    if (!x || !z || !a || !b || !state || !out)
        return fail(GDN_ERR_INVALID_ARG, fn, "an input or output pointer is NULL");
    if (!aligned16(x) || !aligned16(z) || !aligned16(out) || !aligned16(state))
        return fail(GDN_ERR_INVALID_ARG, fn, "x, z, out and the state must be 16-byte aligned");
    if ((st = injected("verify", fn)) != GDN_OK) return st;
    const bool bf16 = dims->dtype == GDN_DTYPE_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gdn::RecurrentArgs r{};
    r.n_seq = n_seq; r.n_k_heads = dims->n_k_heads; r.n_v_heads = dims->n_v_heads;
    r.conv_k = dims->conv_k; r.act = dims->act; r.l2_eps = dims->l2_eps; r.rms_eps = dims->rms_eps;
    r.head_map = dims->head_map; r.decay_form = dims->decay_form;
    r.per_channel = dims->decay_per_channel;
    r.cu_seqlens = nullptr; r.uniform_T = T;
    r.x = x; r.z = z; r.a = a; r.b = b;
    r.conv_w = params->conv_w; r.A_log = params->A_log; r.dt_bias = params->dt_bias;
    r.norm_w = params->norm_w; r.conv_state_in = conv_state;
    r.state_in = state;  // read once; no state, intermediate or history is written
    r.out = out;
    return cuda_status(timed_launch("recurrent", s, [&] {
                           return gdn::launch_recurrent(r, dims->d_k, dims->d_v, bf16, s);
                       }), fn, "recurrent launch");
}

gdn_status gdn_decode_commit(const gdn_dims* dims, int32_t n_seq, int32_t T,
                             const int32_t* accepted, const void* x, const float* inter_states,
                             float* state, void* conv_state, void* stream) {
    const char* fn = "gdn_decode_commit";
    gdn_status st;
    if ((st = check_dims(dims, fn)) != GDN_OK) return st;
    if (n_seq < 0 || n_seq > GDN_MAX_SEQUENCES)
        return fail(GDN_ERR_INVALID_ARG, fn, "n_seq must be 0..GDN_MAX_SEQUENCES (%d) (got %d)",
                    GDN_MAX_SEQUENCES, n_seq);
    if (T < 1 || T > 16) return fail(GDN_ERR_INVALID_ARG, fn, "T must be 1..16 (got %d)", T);
    g_err[0] = '\0';
    if (n_seq == 0) return GDN_OK;
    if (!accepted || !inter_states || !state || (conv_state && !x))
        return fail(GDN_ERR_INVALID_ARG, fn, "a required pointer is NULL");
    if (!aligned16(inter_states) || !aligned16(state))
        return fail(GDN_ERR_INVALID_ARG, fn, "the states must be 16-byte aligned");
    if ((st = injected("commit", fn)) != GDN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gdn::CommitArgs c{};
    c.n_seq = n_seq; c.n_v_heads = dims->n_v_heads; c.d_k = dims->d_k; c.d_v = dims->d_v;
    c.T = T; c.accepted = accepted; c.inter = inter_states; c.state = state;
    if ((st = cuda_status(timed_launch("commit_state", s, [&] { return gdn::launch_commit_state(c, s); }), fn, "commit launch")) != GDN_OK) return st;
    if (conv_state) {
        gdn::ConvStateArgs cs{};
        cs.n_seq = n_seq; cs.n_k_heads = dims->n_k_heads; cs.n_v_heads = dims->n_v_heads;
        cs.d_k = dims->d_k; cs.d_v = dims->d_v; cs.conv_k = dims->conv_k;
        cs.cu_seqlens = nullptr; cs.uniform_T = T; cs.lengths = accepted; cs.x = x;
        cs.conv_state_in = conv_state; cs.conv_state_out = conv_state;
        if ((st = cuda_status(timed_launch("conv_state", s, [&] { return gdn::launch_conv_state(cs, dims->dtype == GDN_DTYPE_BF16, s); }), fn,
                              "conv state launch")) != GDN_OK)
            return st;
    }
    return GDN_OK;
}

}  // extern "C"
