// Status word access and status strings of the C ABI.
#include <cuda_runtime.h>
#include <math.h>

#include <vector>

#include "specv_common.cuh"
#include "specv_trace.h"

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

namespace {

// Self-test of the bounded mbarrier wait that the streaming kernel relies on:
// slot 0 waits on a barrier that nothing completes (the wait must give up
// after limit_ns and report SPEC_ERR_TIMEOUT), slot 1 on one whose phase has
// completed (the wait must succeed at once).
__global__ void k_wait_selftest(unsigned long long limit_ns, int32_t* status, unsigned long long* elapsed_ns) {
    __shared__ __align__(8) uint64_t bars[2];
    if (threadIdx.x != 0) return;
    specv::mbar_init(&bars[0], 1);
    specv::mbar_init(&bars[1], 1);
    specv::fence_mbar_init();
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(specv::smem_u32(&bars[1])) : "memory");
    for (int i = 0; i < 2; ++i) {
        const unsigned long long t0 = specv::globaltimer_ns();
        const bool done = specv::mbar_wait_bounded(&bars[i], 0, limit_ns);
        elapsed_ns[i] = specv::globaltimer_ns() - t0;
        status[i] = done ? SPEC_OK : SPEC_ERR_TIMEOUT;
    }
}

}  // namespace

extern "C" int spec_selftest_wait(long long limit_ns, int32_t* status, unsigned long long* elapsed_ns,
                                  spec_stream_t stream) {
    if (limit_ns < 1000 || limit_ns > 2000000000ll) return SPEC_ERR_SHAPE;
    if (!status || !elapsed_ns) return SPEC_ERR_NULL;
    if (((uintptr_t)status & 3) || ((uintptr_t)elapsed_ns & 7)) return SPEC_ERR_ALIGN;
    k_wait_selftest<<<1, 32, 0, (cudaStream_t)stream>>>((unsigned long long)limit_ns, status, elapsed_ns);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Sequential Temperature Scaling fit on the host ("UraionSpec" §2.4, §3.6).
int spec_sts_fit(const float* confidence, const int32_t* accept_len, int n, int gamma, float* out_temperature,
                 double* out_ece) {
    specv::TraceRange tr("spec_sts_fit");
    if (n < 1 || gamma < 1 || gamma > SPEC_MAX_GAMMA) return SPEC_ERR_SHAPE;
    if (!confidence || !accept_len || !out_temperature) return SPEC_ERR_NULL;
    for (long long i = 0; i < (long long)n * gamma; ++i)
        if (!(confidence[i] >= 0.0f && confidence[i] <= 1.0f)) return SPEC_ERR_CONFIDENCE;
    constexpr int kGrid = 100, kBins = 15;
    std::vector<double> survived(n, 1.0);  // prod over calibrated earlier positions
    std::vector<double> pred(n);
    double in_bin_pred[kBins], in_bin_label[kBins];
    for (int k = 1; k <= gamma; ++k) {
        double best_err = INFINITY, best_t = 1.0;
        for (int g = 0; g < kGrid; ++g) {
            const double t = (double)(g + 1) / 10.0;  // 0.1, 0.2, ..., 10.0
            for (int i = 0; i < n; ++i) pred[i] = survived[i] * pow((double)confidence[(size_t)i * gamma + k - 1], 1.0 / t);
            for (int q = 0; q < kBins; ++q) in_bin_pred[q] = in_bin_label[q] = 0.0;
            for (int i = 0; i < n; ++i) {
                int q = (int)(pred[i] * (double)kBins);
                q = q < 0 ? 0 : (q >= kBins ? kBins - 1 : q);
                in_bin_pred[q] += pred[i];
                in_bin_label[q] += accept_len[i] >= k ? 1.0 : 0.0;
            }
            double err = 0.0;
            for (int q = 0; q < kBins; ++q) err += fabs(in_bin_pred[q] - in_bin_label[q]);
            err /= (double)n;
            if (err < best_err) {
                best_err = err;
                best_t = t;
            }
        }
        out_temperature[k - 1] = (float)best_t;
        if (out_ece) out_ece[k - 1] = best_err;
        for (int i = 0; i < n; ++i) survived[i] *= pow((double)confidence[(size_t)i * gamma + k - 1], 1.0 / best_t);
    }
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
        case SPEC_ERR_ROW_INDEX: return "packed rows of a request lie outside the packed arrays";
        default: return "unknown status";
    }
}

}  // extern "C"
