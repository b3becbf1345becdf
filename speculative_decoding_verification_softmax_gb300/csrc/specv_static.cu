// spec_verify_static: batched verification without a caller-provided
// workspace.
//
// spec_verify needs a few megabytes of device scratch (per-chunk partial sums,
// per-request state, residual chunk sums).  Most callers allocate it once with
// their framework's allocator.  Some callers cannot allocate device memory at
// the point where they verify: code running under an allocator that forbids
// new allocations during a capture or a latency-critical loop, plugins that
// receive only input and output buffers from a host engine, or embedded
// runtimes with a fixed memory budget set at start-up.  For them this file
// keeps one statically sized scratch array in device memory, created when the
// library is loaded on a GPU and held until the process exits.
#include <cuda_runtime.h>

#include "specv_common.cuh"

namespace {

// The shared scratch: SPEC_STATIC_WORKSPACE_BYTES on every device that loads
// the library.  Host code must not use this name as a device address; the
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[SPEC_STATIC_WORKSPACE_BYTES];

// The device address of the static scratch array on the current device.  It
// is looked up on every call (a host-side table lookup once the module is
// loaded), so that an address never outlives the context it belongs to: after
// cudaDeviceReset the module is loaded again and the array may move.  The
// first lookup on a device may load the module, which is why the first call
// belongs before any stream capture.
int static_workspace(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return SPEC_ERR_CUDA;
    *out = p;
    return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_static(const void* target_logits, const void* draft_logits, spec_dtype dt, int B,
                                  int gamma, int V, const int32_t* draft_tokens, const int32_t* verify_len,
                                  float temperature, const float* uniforms, int32_t* out_tokens,
                                  int32_t* out_accept_len, spec_stream_t stream) {
    const size_t need = spec_verify_workspace_bytes(B, gamma, V, dt);
    if (need == 0) return SPEC_ERR_SHAPE;
    if (need > SPEC_STATIC_WORKSPACE_BYTES) return SPEC_ERR_WORKSPACE;
    if (B == 0) return SPEC_OK;
    void* ws = nullptr;
    const int rc = static_workspace(&ws);
    if (rc != SPEC_OK) return rc;
    // Nothing in the scratch has to start at zero: every call writes each word
    // it later reads (the streaming kernel resets the status words itself).
    return spec_verify(target_logits, draft_logits, dt, B, gamma, V, draft_tokens, verify_len, temperature,
                       uniforms, out_tokens, out_accept_len, ws, SPEC_STATIC_WORKSPACE_BYTES, stream);
}
