// gdn_prefill_chunks_noalloc: the single-session prefill with its scratch in
// a fixed array that the library itself owns, for callers that cannot
// allocate device memory.
//
// Who needs it: code whose device memory is planned once, up front, by a host
// framework that owns the allocator (plugin interfaces of inference runtimes
// hand a kernel only the buffers the framework planned), and latency-critical
// callers that must not call cudaMalloc / cudaFree because those calls can
// synchronise the device and stall every other stream. Such callers still
// pass their inputs, outputs and session buffers; only the per-call scratch
// moves into the library.
//
// The scratch is the file-scope array below. Every GPU that loads the library
// holds GDN_NOALLOC_SCRATCH_BYTES of it until the process exits. Host code
// never uses the array's name as an address (on the host it is only a
// stand-in): the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device.
#include "gdn.h"
#include "common.cuh"

#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up on first use).
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) gdn_status gdn_prefill_chunks_noalloc(
    const gdn_layer_desc *desc, gdn_session *session, const void *xq, const void *xk, const void *xv,
    const float *g, const float *beta, const void *conv_w, int64_t n_tokens, uint32_t flags, void *out,
    int64_t *n_consumed, gdn_stream_t stream) {
    gdn_status st = gdn_desc_check(desc);
    if (st != GDN_OK) return st;
    if (n_tokens < 0 || (flags & ~GDN_ALLOW_PARTIAL))   // let the regular validation report it
        return gdn_prefill_chunks(desc, session, xq, xk, xv, g, beta, conv_w, n_tokens, flags, out, n_consumed,
                                  nullptr, 0, stream);
    // Size limit, checked before any CUDA call. gdn_workspace_size(desc, n, 1) counts ceil(n / 64) blocks
    // plus one spare block per launch. The prefill's own check counts ceil(n / 64) blocks for this call,
    // because a call's 64-token blocks start at its first token whether or not the session sits on the
    // grid (a partial call after an off-grid commit included), so a call that passes this check passes that
    // one with the spare block to spare.
    const int64_t processed = (flags & GDN_ALLOW_PARTIAL) ? n_tokens : n_tokens / desc->grid_c * desc->grid_c;
    const size_t need = gdn_workspace_size(desc, processed, 1);
    if (processed > 0 && need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gdn_prefill_chunks_noalloc: %lld tokens need %zu bytes of scratch, above the built-in %u bytes; "
                 "use gdn_prefill_chunks with a caller workspace or split the call",
                 (long long)processed, need, (unsigned)GDN_NOALLOC_SCRATCH_BYTES);
        gdn_internal_set_error(msg);
        return GDN_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "gdn_prefill_chunks_noalloc: scratch address lookup: %s", cudaGetErrorString(e));
        gdn_internal_set_error(msg);
        return GDN_ERR_CUDA;
    }
    // Every element of the scratch this call reads is written earlier in the
    // same call, so the previous call's contents need no clearing.
    return gdn_prefill_chunks(desc, session, xq, xk, xv, g, beta, conv_w, n_tokens, flags, out, n_consumed, scratch,
                              GDN_NOALLOC_SCRATCH_BYTES, stream);
}
