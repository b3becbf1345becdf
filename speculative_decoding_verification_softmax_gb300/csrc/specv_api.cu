// Status word access and status strings of the C ABI.
#include <cuda_runtime.h>

#include "specv_common.cuh"

extern "C" {

int spec_read_status(void* workspace, spec_stream_t stream, int* status) {
    if (!workspace || !status) return SPEC_ERR_NULL;
    cudaStream_t st = (cudaStream_t)stream;
    int v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return SPEC_ERR_CUDA;
    *status = v;
    return SPEC_OK;
}

const char* spec_status_string(int status) {
    switch (status) {
        case SPEC_OK: return "ok";
        case SPEC_ERR_NULL: return "a required pointer is NULL";
        case SPEC_ERR_SHAPE: return "B, gamma, V or min_len out of range";
        case SPEC_ERR_ALIGN: return "a pointer is not aligned to its element size (workspace: 16 bytes)";
        case SPEC_ERR_TEMPERATURE: return "temperature must be 0 or in [1e-4, 1e4]";
        case SPEC_ERR_VERIFY_LEN: return "verify_len outside [0, gamma]";
        case SPEC_ERR_TOKEN: return "draft token id outside [0, V)";
        case SPEC_ERR_WORKSPACE: return "workspace too small";
        case SPEC_ERR_COST_TABLE: return "invalid cost table";
        case SPEC_ERR_NONFINITE: return "a needed logit row has a NaN, +inf or no finite value";
        case SPEC_ERR_TIMEOUT: return "a bounded device wait expired";
        case SPEC_ERR_CUDA: return "CUDA runtime error";
        case SPEC_ERR_UNIFORM: return "a used uniform is outside [0, 1)";
        case SPEC_ERR_CONFIDENCE: return "a confidence is outside [0, 1]";
        default: return "unknown status";
    }
}

}  // extern "C"
