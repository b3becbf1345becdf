// Confidence-scheduled verify lengths on GB300, one CTA per call.
//
// Method (restated from the pages):
//   * Prefix survival s_{b,0} = 1, s_{b,k} = prod_{t<=k} c_{b,t} ("AngelSpec"
//     §4.2, eq. (20)) and estimated progress A_b(n) = sum_{k<=n} s_{b,k}
//     (eq. (21)).
//   * Candidates (b, k > min_len) ordered by survival, ties to the shallower
//     position then the lower request (top-K with shallow-first ties keeps
//     every request's kept drafts a contiguous prefix, §4.2).
//   * Budget N = sum_b (ell_b + 1) ("AngelSpec" §4.1): taking the first
//     N - B(min_len+1) candidates gives the best estimated progress tau(N) for
//     that budget; the call returns the allocation of the first N that
//     maximises tau(N) / C(N) (eq. (24) with every budget a candidate), or,
//     in Algorithm-1 mode ("UraionSpec" §3.5), stops at the first candidate
//     that does not strictly improve tau / C.
//
// All arithmetic is fp64 through explicit round-to-nearest intrinsics, in a
// fixed order (products and sums left to right, tau summed sequentially in
// sorted order), so the result is reproducible bit for bit.
#include <math.h>
#include <stdint.h>

#include "specv_common.cuh"

namespace specv {

struct SchedArgs {
    const float* conf;
    int32_t* out;
    int* status;
    int B, gamma, min_len, mode, nk, nc, npad;
    int has_sts;
    double kt[32];
    double kc[32];
    float sts[32];  // STS temperatures per position (has_sts)
};

// Confidence of position k (1-based), calibrated by c^(1/T_k) when STS
// temperatures are given ("UraionSpec" §2.4).
__device__ __forceinline__ double conf_at(const float* conf, const float* sts, int has_sts, size_t i, int k) {
    const double c = (double)conf[i];
    return has_sts ? pow(c, __ddiv_rn(1.0, (double)sts[k - 1])) : c;
}

__device__ __forceinline__ double cost_at(double N, const SchedArgs& a) {
    if (N <= a.kt[0]) return a.kc[0];
    if (N >= a.kt[a.nk - 1]) return a.kc[a.nk - 1];
    int i = 0;
    while (!(N < a.kt[i + 1])) ++i;
    return __dadd_rn(a.kc[i], __ddiv_rn(__dmul_rn(__dsub_rn(N, a.kt[i]), __dsub_rn(a.kc[i + 1], a.kc[i])),
                                        __dsub_rn(a.kt[i + 1], a.kt[i])));
}

__global__ void __launch_bounds__(1024) k_schedule(SchedArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 15) & ~uintptr_t(15));
    unsigned long long* key = (unsigned long long*)smem;          // [npad]; later tau / objectives
    unsigned* id = (unsigned*)(key + a.npad);                    // [npad]
    double* prog = (double*)(((uintptr_t)(id + a.npad) + 7) & ~uintptr_t(7));  // [B]; later counts
    __shared__ int s_bad, s_npos, s_dcut_k;
    __shared__ double s_base;
    __shared__ double s_red_v[32];
    __shared__ int s_red_i[32];

    const int tid = threadIdx.x, nt = blockDim.x;
    const int B = a.B, G = a.gamma, ml = a.min_len, per = G - ml;
    if (tid == 0) {
        s_bad = 0;
        *a.status = 0;
    }
    __syncthreads();
    for (int i = tid; i < B * G; i += nt) {
        const float c = a.conf[i];
        if (!(c >= 0.0f && c <= 1.0f)) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        for (int b = tid; b < B; b += nt) a.out[b] = -1;
        if (tid == 0) *a.status = SPEC_ERR_CONFIDENCE;
        return;
    }

    // survival products, progress at min_len, candidate keys
    for (int b = tid; b < B; b += nt) {
        double s = 1.0, A = __dadd_rn(0.0, 1.0);
        for (int k = 1; k <= G; ++k) {
            s = __dmul_rn(s, conf_at(a.conf, a.sts, a.has_sts, (size_t)b * G + k - 1, k));
            if (k <= ml) {
                A = __dadd_rn(A, s);
            } else {
                const int ci = b * per + (k - ml - 1);
                key[ci] = ~(unsigned long long)__double_as_longlong(s);
                id[ci] = ((unsigned)k << 12) | (unsigned)b;
            }
        }
        prog[b] = A;
    }
    for (int i = a.nc + tid; i < a.npad; i += nt) {
        key[i] = ~0ull;
        id[i] = ~0u;
    }
    __syncthreads();
    if (tid == 0) {
        double base = 0.0;
        for (int b = 0; b < B; ++b) base = __dadd_rn(base, prog[b]);
        s_base = base;
    }

    // bitonic sort ascending on (key, id): survival descending, then k, then b
    for (int k = 2; k <= a.npad; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            __syncthreads();
            for (int i = tid; i < a.npad; i += nt) {
                const int p = i ^ j;
                if (p > i) {
                    const unsigned long long ki = key[i], kp = key[p];
                    const unsigned ii = id[i], ip = id[p];
                    const bool gt = ki > kp || (ki == kp && ii > ip);
                    if (gt == ((i & k) == 0)) {
                        key[i] = kp;
                        key[p] = ki;
                        id[i] = ip;
                        id[p] = ii;
                    }
                }
            }
        }
    }
    __syncthreads();

    // tau(N0 + i + 1) summed sequentially in sorted order
    const double N0 = __dmul_rn((double)B, (double)(ml + 1));
    if (tid == 0) {
        s_dcut_k = 0;
        double tau = s_base;
        int npos = a.nc;
        for (int i = 0; i < a.nc; ++i) {
            const double s = __longlong_as_double((long long)~key[i]);
            if (npos == a.nc && !(s > 0.0)) npos = i;
            tau = __dadd_rn(tau, s);
            key[i] = (unsigned long long)__double_as_longlong(tau);
        }
        s_npos = npos;
        if (a.mode == SPEC_SCHED_DCUT) {
            // D-cut: tau at the budgets K_i = max(N0, ceil(rho_i * B(gamma+1))), first max of tau / C_i
            const double Nmax = __dmul_rn((double)B, (double)(G + 1));
            double best = -INFINITY;
            int bestK = 0;
            for (int i = 0; i < a.nk; ++i) {
                double K = ceil(__dmul_rn(a.kt[i], Nmax));
                if (K < N0) K = N0;
                if (K > Nmax) K = Nmax;
                const int take = (int)__dsub_rn(K, N0);
                const double tau = take == 0 ? s_base : __longlong_as_double((long long)key[take - 1]);
                const double obj = __ddiv_rn(tau, a.kc[i]);
                if (obj > best) {
                    best = obj;
                    bestK = take;
                }
            }
            s_dcut_k = bestK;
        }
    }
    __syncthreads();
    // objectives: obj(K) for K = 1..nc in key[K-1]; obj(0) from the base
    for (int i = tid; i < a.nc; i += nt) {
        const double tau = __longlong_as_double((long long)key[i]);
        key[i] = (unsigned long long)__double_as_longlong(
            __ddiv_rn(tau, cost_at(__dadd_rn(N0, (double)(i + 1)), a)));
    }
    __syncthreads();
    const double obj0 = __ddiv_rn(s_base, cost_at(N0, a));
    auto obj = [&](int K) -> double { return K == 0 ? obj0 : __longlong_as_double((long long)key[K - 1]); };

    // pick K: exact = first maximum; Algorithm 1 = first non-improving valid candidate
    double bv = -INFINITY;
    int bi = 0x7fffffff;
    if (a.mode == SPEC_SCHED_EXACT) {
        for (int K = tid; K <= a.nc; K += nt) {
            const double v = obj(K);
            if (v > bv || (v == bv && K < bi)) { bv = v; bi = K; }
        }
    } else {
        bv = 0.0;
        for (int i = tid; i < s_npos; i += nt)
            if (!(obj(i + 1) > obj(i)) && i < bi) bi = i;
        if (tid == 0 && s_npos < bi) bi = s_npos;
    }
    const int lane = tid & 31, warp = tid >> 5;
    for (int o = 16; o > 0; o >>= 1) {
        const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) {
        s_red_v[warp] = bv;
        s_red_i[warp] = bi;
    }
    int* count = (int*)prog;
    for (int b = tid; b < B; b += nt) count[b] = 0;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        bv = lane < nw ? s_red_v[lane] : -INFINITY;
        bi = lane < nw ? s_red_i[lane] : 0x7fffffff;
        for (int o = 16; o > 0; o >>= 1) {
            const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) s_red_i[0] = bi;
    }
    __syncthreads();
    const int bestK = a.mode == SPEC_SCHED_DCUT ? s_dcut_k : s_red_i[0];
    for (int i = tid; i < bestK; i += nt) atomicAdd(&count[id[i] & 4095u], 1);
    __syncthreads();
    for (int b = tid; b < B; b += nt) a.out[b] = ml + count[b];
}

// Static verify lengths: the leading positions whose (calibrated) confidence
// is at least the threshold, clamped to [min_len, max_len].  One thread per
// request.
__global__ void k_schedule_static(const float* conf, int B, int G, double threshold, int max_len, int min_len,
                                  int has_sts, SchedArgs sa, int32_t* out, int* status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int n = 0;
    bool bad = false;
    if (threshold <= 0.0) {
        n = max_len;
        if (conf)
            for (int k = 0; k < G; ++k) {
                const float c = conf[(size_t)b * G + k];
                bad |= !(c >= 0.0f && c <= 1.0f);
            }
    } else {
        for (int k = 0; k < G; ++k) {
            const float c = conf[(size_t)b * G + k];
            bad |= !(c >= 0.0f && c <= 1.0f);
        }
        while (!bad && n < max_len && conf_at(conf, sa.sts, has_sts, (size_t)b * G + n, n + 1) >= threshold) ++n;
    }
    if (bad) {
        out[b] = -1;
        atomicCAS(status, 0, SPEC_ERR_CONFIDENCE);
        return;
    }
    out[b] = n < min_len ? min_len : n;
}

}  // namespace specv

using namespace specv;

namespace {
bool g_sched_attr[64];
}

extern "C" {

size_t spec_schedule_workspace_bytes(int B, int gamma) {
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA) return 0;
    return 256;
}

static bool sts_ok(const float* T, int gamma) {
    if (!T) return true;
    for (int k = 0; k < gamma; ++k)
        if (!(T[k] > 0.0f) || !isfinite(T[k])) return false;
    return true;
}

int spec_schedule(const float* confidence, int B, int gamma, const spec_cost_table* cost, int min_len,
                  spec_sched_mode mode, const float* sts_temperature, int32_t* out_verify_len, void* workspace,
                  size_t workspace_bytes, spec_stream_t stream) {
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA || min_len < 0 || min_len > gamma)
        return SPEC_ERR_SHAPE;
    if ((long long)B * (gamma - min_len) > SPEC_MAX_SCHED_CANDIDATES) return SPEC_ERR_SHAPE;
    if (mode != SPEC_SCHED_EXACT && mode != SPEC_SCHED_ALGORITHM1 && mode != SPEC_SCHED_DCUT) return SPEC_ERR_SHAPE;
    if (!cost) return SPEC_ERR_NULL;
    if (cost->n < 1 || cost->n > 32) return SPEC_ERR_COST_TABLE;
    for (int i = 0; i < cost->n; ++i) {
        if (!isfinite(cost->tokens[i]) || !isfinite(cost->cost_ms[i]) || !(cost->cost_ms[i] > 0.0))
            return SPEC_ERR_COST_TABLE;
        if (i > 0 && !(cost->tokens[i] > cost->tokens[i - 1])) return SPEC_ERR_COST_TABLE;
        if (mode == SPEC_SCHED_DCUT && !(cost->tokens[i] > 0.0 && cost->tokens[i] <= 1.0)) return SPEC_ERR_COST_TABLE;
    }
    if (!sts_ok(sts_temperature, gamma)) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;
    if (!out_verify_len || !workspace || (gamma > 0 && !confidence)) return SPEC_ERR_NULL;
    if (((uintptr_t)out_verify_len & 3) || ((uintptr_t)workspace & 15) || ((uintptr_t)confidence & 3))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < 256) return SPEC_ERR_WORKSPACE;

    SchedArgs a;
    a.conf = confidence;
    a.out = out_verify_len;
    a.status = (int*)workspace;
    a.B = B;
    a.gamma = gamma;
    a.min_len = min_len;
    a.mode = (int)mode;
    a.nk = cost->n;
    a.nc = B * (gamma - min_len);
    int npad = 1;
    while (npad < a.nc) npad <<= 1;
    a.npad = npad;
    for (int i = 0; i < 32; ++i) {
        a.kt[i] = i < cost->n ? cost->tokens[i] : 0.0;
        a.kc[i] = i < cost->n ? cost->cost_ms[i] : 0.0;
        a.sts[i] = (sts_temperature && i < gamma) ? sts_temperature[i] : 1.0f;
    }
    a.has_sts = sts_temperature ? 1 : 0;
    const size_t smem = (size_t)npad * 12 + (size_t)B * 8 + 32;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    if (!g_sched_attr[dev]) {
        const int max_smem = SPEC_MAX_SCHED_CANDIDATES * 12 + SPEC_MAX_BATCH * 8 + 32;
        if (cudaFuncSetAttribute((const void*)k_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 max_smem) != cudaSuccess)
            return SPEC_ERR_CUDA;
        g_sched_attr[dev] = true;
    }
    k_schedule<<<1, 1024, smem, (cudaStream_t)stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int spec_schedule_static(const float* confidence, int B, int gamma, float threshold, int max_len, int min_len,
                         const float* sts_temperature, int32_t* out_verify_len, void* workspace,
                         size_t workspace_bytes, spec_stream_t stream) {
    if (B < 0 || B > SPEC_MAX_BATCH || gamma < 0 || gamma > SPEC_MAX_GAMMA || min_len < 0 || min_len > max_len ||
        max_len > gamma)
        return SPEC_ERR_SHAPE;
    if (!(threshold == threshold)) return SPEC_ERR_SHAPE;
    if (!sts_ok(sts_temperature, gamma)) return SPEC_ERR_SHAPE;
    if (B == 0) return SPEC_OK;
    if (!out_verify_len || !workspace || (threshold > 0.0f && gamma > 0 && !confidence)) return SPEC_ERR_NULL;
    if (((uintptr_t)out_verify_len & 3) || ((uintptr_t)workspace & 15) || ((uintptr_t)confidence & 3))
        return SPEC_ERR_ALIGN;
    if (workspace_bytes < 256) return SPEC_ERR_WORKSPACE;
    SchedArgs sa;
    for (int i = 0; i < 32; ++i) sa.sts[i] = (sts_temperature && i < gamma) ? sts_temperature[i] : 1.0f;
    // The status word is cleared before the launch: a block that finds a bad
    // confidence may finish before any other block starts.
    if (cudaMemsetAsync(workspace, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess) return SPEC_ERR_CUDA;
    k_schedule_static<<<(B + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
        gamma > 0 ? confidence : nullptr, B, gamma, (double)threshold, max_len, min_len, sts_temperature ? 1 : 0, sa,
        out_verify_len, (int*)workspace);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
