// gdn_prefill_noalloc: the prefill for callers that cannot allocate device
// memory.  Some hosts of this core run it where no allocation may happen: an
// inference engine's plugin that is handed its inputs and outputs but no
// workspace, or a serving loop that has fixed its memory before the first
// request.  Such a caller cannot size and pass the scratch memory that
// gdn_prefill asks for, so this entry point brings its own: one file-scope
// device array.  It becomes resident on a device when this module is loaded
// there; under CUDA's default lazy module loading that is the first
// gdn_prefill_noalloc call on the device (its cudaGetSymbolAddress), which is
// why that call belongs in the caller's set-up.  It then stays resident until
// the process exits.
//
// Nothing here allocates: no cudaMalloc, cudaFree or allocating library
// routine.  The array's device address is looked up once per device with
// cudaGetSymbolAddress (host code cannot use the array's name as a device
// address: on the host that name is only a stand-in), and the call then runs
// the regular prefill with that address as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {
// Records the thread's error message (defined with the other entry points).
gdn_status set_error(gdn_status st, const char* fn, const char* fmt, ...);
}  // namespace gdn

namespace {

// 64 MiB: the chunked tensor-core prefill of a few hundred tokens at
// Hk = 16, Hv = 32, d_k = d_v = 128 (about 107 KB per token).
constexpr size_t kPrefillScratchBytes = size_t(64) << 20;

// Shared by every call on a device; keeps the last call's contents.  Every
// region the prefill reads is written earlier in the same call (rows of a
// partial chunk past its end are masked when loaded), so nothing needs to be
// cleared between calls.
static __device__ __align__(256) unsigned char g_prefill_scratch[kPrefillScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the
// first call for that device and kept (like the library's other per-device
// state, it assumes the device's primary context lives as long as the process;
// a cudaDeviceReset voids it).
gdn_status scratch_address(void** ptr, const char* fn) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return gdn::set_error(GDN_ERR_CUDA, fn, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return gdn::set_error(GDN_ERR_UNSUPPORTED, fn, "device %d is beyond the %d this call serves",
                              dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess || !p)
            return gdn::set_error(GDN_ERR_CUDA, fn, "cudaGetSymbolAddress of the scratch failed: %s",
                                  cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" size_t gdn_prefill_noalloc_scratch_bytes(void) { return kPrefillScratchBytes; }

extern "C" gdn_status gdn_prefill_noalloc(const gdn_dims* dims, const gdn_params* params,
                                          int32_t n_seq, const int32_t* cu_seqlens,
                                          const int32_t* cu_seqlens_host, const void* x,
                                          const void* z, const void* a, const void* b,
                                          const void* conv_state_in, void* conv_state_out,
                                          const float* initial_state, float* final_state,
                                          void* out, void* stream) {
    const char* fn = "gdn_prefill_noalloc";
    size_t need = 0;
    gdn_status st = gdn_prefill_workspace_size(dims, n_seq, cu_seqlens_host, &need);
    if (st != GDN_OK) return st;
    if (need > kPrefillScratchBytes)
        return gdn::set_error(GDN_ERR_WORKSPACE, fn,
                              "this sequence layout needs %zu bytes of scratch but the built-in "
                              "scratch holds %zu; use gdn_prefill with a caller workspace",
                              need, kPrefillScratchBytes);
    void* scratch = nullptr;
    if (need > 0 && (st = scratch_address(&scratch, fn)) != GDN_OK) return st;
    return gdn_prefill(dims, params, n_seq, cu_seqlens, cu_seqlens_host, x, z, a, b,
                       conv_state_in, conv_state_out, initial_state, final_state, out, scratch,
                       need > 0 ? kPrefillScratchBytes : 0, stream);
}
