// Shared device helpers of the verification and scheduling kernels:
// inline PTX for mbarriers, 1-D bulk copies (cp.async.bulk), NaN-propagating
// max, the MUFU base-2 exponential, warp reductions, and the workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/specv.h"

namespace specv {

// ---------------------------------------------------------------- tunables
// Bytes of one row chunk: the unit of work of one warp in the streaming pass
// and of the residual pass.  4 KiB = 2048 bf16 or 1024 fp32 logits.
constexpr int kChunkBytes = 4096;
// Row-statistics kernel: warps per CTA and bulk-copy stages per warp.
constexpr int kStatsWarps = 20;
constexpr int kStages = 2;
// Bound on any device wait (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// Largest grid of the streaming kernel (one word per CTA in the workspace,
// read by the finish kernel's first warp as two 16-byte vectors per lane).
constexpr int kMaxStatsGrid = 256;

// ----------------------------------------------------------- workspace
// Per-request state written by the accept kernel, read by the draw kernel.
struct ReqState {
    int ell;     // verify length (valid only when status == SPEC_OK)
    int status;  // SPEC_OK or a device error code
    int n;       // accepted drafts
    int mode;    // 0: nothing to draw, 1: residual draw, 2: bonus draw
    int g_t;     // global row id of the target row of the draw
    int g_d;     // global row id of the draft row (residual) or -1
    float u;     // uniform of the draw
    float M_t;   // integer row scale of the target draw row
    float M_d;   // integer row scale of the draft draw row
    float rho_hi, rho_lo;  // S_t / S_d as an unevaluated float pair
    float S_hi, S_lo;      // row sum of the target draw row, unevaluated float pair
};

// Unevaluated sum hi + lo of two floats (about 48 significant bits).
struct DF {
    float hi, lo;
};

// (a + b) with the rounding error carried (Knuth's TwoSum, then renormalised).
__device__ __forceinline__ DF df_add(DF a, DF b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float err = (a.hi - (s - bb)) + (b.hi - bb);
    const float lo = err + a.lo + b.lo;
    DF r;
    r.hi = s + lo;
    r.lo = lo - (r.hi - s);
    return r;
}

__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        DF w;
        w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = df_add(v, w);
    }
    return v;
}

// a / b for two-float numbers (one correction step; about 44 significant bits).
__device__ __forceinline__ DF df_div(DF a, DF b) {
    const float q = a.hi / b.hi;
    // remainder a - q * b, the product q * b.hi carried exactly by an fma
    const float p = q * b.hi;
    const float pe = fmaf(q, b.hi, -p);
    const float rem = ((a.hi - p) - pe) + a.lo - q * b.lo;
    DF r;
    r.hi = q + rem / b.hi;
    r.lo = (q - r.hi) + rem / b.hi;
    return r;
}

// Inclusive warp scan of two-float values (lane order).
__device__ __forceinline__ DF warp_scan_df(DF v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        DF w;
        w.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
        if (lane >= o) v = df_add(w, v);
    }
    return v;
}

__device__ __forceinline__ double df_to_d(DF v) { return (double)v.hi + (double)v.lo; }

// 2^e as a float for integer e <= 0 (0 below the normal range).
__device__ __forceinline__ float pow2_f(int e) {
    return e < -126 ? 0.0f : __int_as_float((127 + e) << 23);
}

struct Layout {
    int R;        // B * (2*gamma + 1) potential rows
    int nch;      // chunks per row
    int CH;       // elements per chunk
    size_t hdr, ctaw, partial, req, pq, mass, rchunk, total;

    __host__ __device__ static size_t up(size_t x) { return (x + 255) & ~size_t(255); }

    __host__ __device__ Layout(int B, int gamma, int V, int es) {
        R = B * (2 * gamma + 1);
        CH = kChunkBytes / es;
        nch = (int)(((long long)V + CH - 1) / CH);
        size_t o = 0;
        hdr = o;      o = up(o + 256);
        ctaw = o;     o = up(o + sizeof(int) * (size_t)kMaxStatsGrid);
        partial = o;  o = up(o + sizeof(float2) * (size_t)R * (size_t)nch);
        req = o;      o = up(o + sizeof(ReqState) * (size_t)B);
        pq = o;       o = up(o + 2 * sizeof(float) * (size_t)B * (size_t)(gamma > 0 ? gamma : 1));
        mass = o;     o = up(o + sizeof(float2) * (size_t)B);
        rchunk = o;   o = up(o + sizeof(float) * (size_t)B * (size_t)nch);
        total = o;
    }
};

// Header words (int32) at the start of the workspace: the status of the most
// recent call (reset by its streaming kernel, set by its finish kernel, read
// and cleared by spec_read_status) and its event bits.  Timeouts of the
// streaming kernel go to one word per CTA (the `ctaw` section), written by
// every CTA of every call, so no CTA's reset can race with another's error.
constexpr int kHdrStatus = 0;
constexpr int kHdrEvents = 2;

// ------------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase `parity` of `bar`; gives up after limit_ns of the
// global timer (monotonic), so the wait always ends.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (tx bytes).
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float c;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(c) : "f"(a), "f"(b));
    return c;
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t c;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(a), "r"(b));
    return c;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Exponent of one logit at scale (c_hi + c_lo) relative to the integer row
// scale M: t = z*c - M, with the product carried as a float pair.  c_lo > 0
// keeps t = -inf for z = -inf.
__device__ __forceinline__ float scaled_exp(float z, float c_hi, float c_lo, float M) {
    return ex2_approx(fmaf(z, c_lo, fmaf(z, c_hi, -M)));
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// allow the next kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Where the logit rows of a request live.  Padded layout (trow == nullptr):
// target row (b, j) is row b*(gamma+1) + j of the target array and draft row
// (b, j) is row b*gamma + j of the draft array.  Packed layout: rows
// trow[b] + j of a [Kt, V] target array and drow[b] + j of a [Kd, V] draft
// array.
struct RowMap {
    const int32_t* trow;
    const int32_t* drow;
    int Kt, Kd;
};

__device__ __forceinline__ size_t target_row(const RowMap& m, int b, int j, int G1) {
    return m.trow ? (size_t)(m.trow[b] + j) : (size_t)b * G1 + j;
}

__device__ __forceinline__ size_t draft_row(const RowMap& m, int b, int j, int G) {
    return m.drow ? (size_t)(m.drow[b] + j) : (size_t)b * G + j;
}

// True when the rows request b reads (target 0..ell, draft 0..ell-1 if
// `draft`) lie inside the packed arrays; always true for the padded layout.
__device__ __forceinline__ bool rows_in_range(const RowMap& m, int b, int ell, bool draft) {
    if (!m.trow) return true;
    const int t = m.trow[b];
    bool ok = t >= 0 && t <= m.Kt - ell - 1;
    if (draft && ell > 0) {
        const int d = m.drow[b];
        ok = ok && d >= 0 && d <= m.Kd - ell;
    }
    return ok;
}

__device__ __forceinline__ void set_status(int* status_word, int err) {
    atomicCAS(status_word, 0, err);
}

// Element range of one chunk of one row, split into an aligned interior that
// is copied or loaded in 16-byte vectors and scalar head / tail elements.
struct ChunkSpan {
    const char* rowp;  // row base
    int e0, e1;        // chunk element range [e0, e1)
    int ia, ib;        // aligned interior [ia, ib); ia == ib == e1 if empty
};

template <int ES>
__device__ __forceinline__ ChunkSpan chunk_span(const char* rowp, int e0, int e1) {
    ChunkSpan s;
    s.rowp = rowp;
    s.e0 = e0;
    s.e1 = e1;
    const uintptr_t p0 = (uintptr_t)(rowp + (size_t)e0 * ES);
    const uintptr_t p1 = (uintptr_t)(rowp + (size_t)e1 * ES);
    const uintptr_t A = (p0 + 15) & ~uintptr_t(15);
    const uintptr_t Z = p1 & ~uintptr_t(15);
    if (Z > A) {
        s.ia = e0 + (int)((A - p0) / ES);
        s.ib = e0 + (int)((Z - p0) / ES);
    } else {
        s.ia = s.ib = e1;
    }
    return s;
}

// The single scalar element a lane handles for a span (head: lanes 0-15,
// tail: lanes 16-31), or -1.  Head <= 15 elements, tail <= 7 (bf16).
__device__ __forceinline__ int span_scalar_index(const ChunkSpan& s, int lane) {
    if (lane < 16) {
        const int i = s.e0 + lane;
        return i < s.ia ? i : -1;
    }
    const int i = s.ib + (lane - 16);
    return (i < s.e1 && s.ib < s.e1 && s.ia < s.ib) ? i : -1;
}

template <int ES>
__device__ __forceinline__ float load_logit(const char* rowp, int i) {
    if (ES == 2) {
        const uint32_t h = *(const unsigned short*)(rowp + (size_t)i * 2);
        return __uint_as_float(h << 16);
    }
    return *(const float*)(rowp + (size_t)i * 4);
}

}  // namespace specv
